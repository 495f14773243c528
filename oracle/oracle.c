/*
 * Oracle for exact scaled dot-product attention, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * CPU definition that the CUDA path is checked against.  Only the test suite,
 * the package smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or helper with the CUDA library, and the
 * library never calls it.
 *
 * Everything is IEEE double.  Inputs of narrower types are widened exactly by
 * the caller before they reach this file.
 *
 * What is computed, and where it is defined:
 *
 *  - Scores and output.  TIGA-lang, "注意力与稠密关系" (attention examples),
 *    section "全量注意力，无掩码" (full attention, no mask), its display
 *    equation:  s_hij = <k_hj, q_hi> * scale,  out_hi = sum_j softmax_j(s) v_hj.
 *    The pages use scale = D^-1/2; here the scale is an argument.
 *
 *  - Relations.  Same page, section "因果稠密关系" (causal dense relation):
 *    query i admits key j iff j <= i.  Section "用图组合表达 varlen 因果注意力"
 *    (varlen causal attention by graph composition): a key is admitted only
 *    inside the query's own sequence, seq(i) = b <=> cu_b <= i < cu_{b+1}.
 *    Positions i, j below are offsets inside the sequence.
 *
 *  - Composed two-pass softmax.  OCANNL "Module Ir.Online_softmax", opening
 *    paragraph: a max-reduction, then a sum of exponentials shifted by that
 *    max, then the reduction against v.  The oracle is exactly that composed
 *    form (probabilities normalised first, then summed against v); it is NOT
 *    the online / block recurrence the GPU path uses.
 *
 *  - Row log-sum-exp.  The final (m, l) of a row, persisted for the backward
 *    (OCANNL page, fourth bullet: "the final (m, l) land in their nodes"),
 *    reported as lse = m + ln l, natural log of the sum over admitted keys of
 *    exp(scaled score).
 *
 *  - Backward.  The textbook softmax Jacobian, written out:
 *        P_ij  = exp(s_ij - m_i) / l_i
 *        dP_ij = <dO_i, v_j>
 *        c_i   = sum_j P_ij dP_ij
 *        dS_ij = P_ij (dP_ij - c_i)
 *        dq_i = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i,
 *        dv_j = sum_i P_ij dO_i.
 *    c_i is computed from P and dP, deliberately not from the shortcut
 *    D_i = <dO_i, O_i> that the OCANNL page's third bullet uses; the tests
 *    check that identity separately.
 *
 * Readings where the pages are silent (also listed in the design notes):
 *  - A row that admits no key (only possible for an empty key segment under
 *    the full relation) gets O = 0 and lse = -inf.
 *  - Causal is defined only for a sequence whose query and key lengths are
 *    equal; other inputs return -1.
 *
 *  - Merge of partial results over disjoint key sets (the split-K forward of
 *    the Vx issue "Chunked-dot Reduce lowering: shorten the reduction
 *    dependency chain", measurement section: split-K with C = 8 key chunks).
 *    Attention over the union of C disjoint key sets, from each set's own
 *    result (O_c, lse_c): softmax over the union weighs set c by
 *    exp(lse_c) / sum_c' exp(lse_c'), so
 *        lse = ln sum_c exp(lse_c),   O = sum_c exp(lse_c - lse) O_c.
 *    This is the (m, l, U) state merge of the OCANNL page's block recurrence
 *    (fourth bullet) with each partial's state written as m_c = lse_c,
 *    l_c = 1, U_c = O_c.  The exponentials are taken relative to
 *    M = max_c lse_c.  A partial with lse_c = -inf admits no key and has
 *    weight 0; if every partial is -inf the row gets O = 0, lse = -inf.
 *
 *  - Tile-pruned approximate attention.  TIGA-lang attention examples page,
 *    section "基于 tile 剪枝的稀疏注意力" (tile-pruned sparse attention),
 *    display equations.  A tile pairs a block of block_q query rows with a
 *    block of block_k keys.  For each query block the key tiles are visited
 *    in order; every tile's scores are computed, and m_tile, the largest
 *    score of the whole tile, is compared with m_run, the largest score of
 *    the tiles admitted so far for this query block (the block's rolling
 *    max).  The tile is admitted iff
 *        m_tile >= m_run + ln(rho),   0 < rho <= 1
 *    (the first tile always is: m_run starts at -inf).  An admitted tile
 *    raises m_run to max(m_run, m_tile); a pruned tile contributes nothing.
 *    Each query row's output is then softmax attention over the keys of its
 *    block's admitted tiles only.  Only the dense (full) relation over one
 *    sequence is defined (the page's other paths fail closed).  Rows past
 *    the end of the queries and keys past the end of the keys are not part
 *    of any tile.
 *
 *  - Attention over a general CSR relation.  TIGA-lang attention examples
 *    page: section "用图组合表达 varlen 因果注意力" (the relation as an explicit
 *    CSR graph holding exactly the admitted edges; a missing edge is simply
 *    absent) and section "用 nn 打分的 GAT 边注意力", its display equation
 *        out_i = sum_{e = (j -> i)} exp(s_e) / sum_{e' = (j' -> i)} exp(s_e') x_j,
 *    a softmax over the incoming edges of each destination row.  Row i's
 *    edges are col[row_ptr[i] .. row_ptr[i+1]); a repeated edge counts once
 *    per occurrence.  The score of an edge is either given per edge and head
 *    (a field score; the page's score network itself is not part of this) or
 *    the dot-product score scale * <q_i, k_j>.  A row without edges gets
 *    O = 0, lse = -inf.
 *
 * Layout: q, o, dq, dO are (T_q, H, D) row-major; k, v, dk, dv are (T_k, H, D);
 * lse is (H, T_q).  cu_q / cu_k hold n_seq + 1 cumulative offsets starting at 0.
 * All arrays are host memory owned by the caller.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_ABI_VERSION 1

int oracle_abi_version(void) { return ORACLE_ABI_VERSION; }

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Segment holding global token index t, by linear scan over the offsets. */
static int segment_of(int n_seq, const int32_t *cu, int64_t t)
{
    for (int b = 0; b < n_seq; ++b)
        if (t >= cu[b] && t < cu[b + 1]) return b;
    return -1;
}

static int check_segments(int n_seq, const int32_t *cu_q, const int32_t *cu_k, int causal)
{
    if (n_seq < 1 || !cu_q || !cu_k) return -1;
    if (cu_q[0] != 0 || cu_k[0] != 0) return -1;
    for (int b = 0; b < n_seq; ++b) {
        if (cu_q[b + 1] < cu_q[b] || cu_k[b + 1] < cu_k[b]) return -1;
        if (causal && (cu_q[b + 1] - cu_q[b]) != (cu_k[b + 1] - cu_k[b])) return -1;
    }
    return 0;
}

/* Number of keys that query offset i of a segment with Lk keys admits. */
static int admitted(int i, int Lk, int causal)
{
    if (!causal) return Lk;
    return i + 1 < Lk ? i + 1 : Lk;
}

static double dot(const double *a, const double *b, int D)
{
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += a[d] * b[d];
    return acc;
}

/*
 * Row statistics of one query row: scores s_j for its nj admitted keys
 * (written to s[]), their max m and the shifted sum l = sum_j exp(s_j - m).
 */
static void row_scores(const double *qi, const double *k0, int64_t ldk, int nj, int D,
                       double scale, double *s, double *m_out, double *l_out)
{
    double m = -INFINITY;
    for (int j = 0; j < nj; ++j) {
        s[j] = scale * dot(qi, k0 + (int64_t)j * ldk, D);
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int j = 0; j < nj; ++j) l += exp(s[j] - m);
    *m_out = m;
    *l_out = l;
}

/* Forward for one (query token, head): O row and lse, by the composed form. */
static void fwd_one(int n_seq, const int32_t *cu_q, const int32_t *cu_k, int H, int D,
                    const double *q, const double *k, const double *v, double scale,
                    int causal, int64_t t, int h, double *o_row, double *lse_out, double *s)
{
    const int b = segment_of(n_seq, cu_q, t);
    const int i = (int)(t - cu_q[b]);
    const int Lk = cu_k[b + 1] - cu_k[b];
    const int nj = admitted(i, Lk, causal);
    const int64_t ld = (int64_t)H * D;
    const double *qi = q + t * ld + (int64_t)h * D;
    const double *k0 = k + (int64_t)cu_k[b] * ld + (int64_t)h * D;
    const double *v0 = v + (int64_t)cu_k[b] * ld + (int64_t)h * D;

    for (int d = 0; d < D; ++d) o_row[d] = 0.0;
    if (nj == 0) {
        *lse_out = -INFINITY;
        return;
    }
    double m, l;
    row_scores(qi, k0, ld, nj, D, scale, s, &m, &l);
    for (int j = 0; j < nj; ++j) {
        const double p = exp(s[j] - m) / l; /* normalised probability first */
        const double *vj = v0 + (int64_t)j * ld;
        for (int d = 0; d < D; ++d) o_row[d] += p * vj[d];
    }
    *lse_out = m + log(l);
}

static int max_len(int n_seq, const int32_t *cu)
{
    int mx = 0;
    for (int b = 0; b < n_seq; ++b)
        if (cu[b + 1] - cu[b] > mx) mx = cu[b + 1] - cu[b];
    return mx;
}

static void set_threads(int n_threads)
{
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
}

/*
 * Full forward: every (query token, head).  o is (T_q, H, D), lse is (H, T_q).
 * Returns 0, or -1 on inconsistent segments.
 */
int oracle_attn_fwd(int n_seq, const int32_t *cu_q, const int32_t *cu_k, int H, int D,
                    const double *q, const double *k, const double *v, double scale,
                    int causal, double *o, double *lse, int n_threads)
{
    if (check_segments(n_seq, cu_q, cu_k, causal) || H < 1 || D < 1) return -1;
    set_threads(n_threads);
    const int64_t Tq = cu_q[n_seq];
    const int Lk_max = max_len(n_seq, cu_k);
    const int64_t n_rows = Tq * H;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Lk_max > 0 ? Lk_max : 1));
#pragma omp for schedule(dynamic, 8)
        for (int64_t r = 0; r < n_rows; ++r) {
            const int64_t t = r / H;
            const int h = (int)(r % H);
            fwd_one(n_seq, cu_q, cu_k, H, D, q, k, v, scale, causal, t, h,
                    o + r * D, lse + (int64_t)h * Tq + t, s);
        }
        free(s);
    }
    return 0;
}

/*
 * Sampled forward: only the listed (token, head) query rows.  o_rows is
 * (n, D), lse_rows is (n).  Used to check full-size runs row by row.
 */
int oracle_attn_fwd_rows(int n_seq, const int32_t *cu_q, const int32_t *cu_k, int H, int D,
                         const double *q, const double *k, const double *v, double scale,
                         int causal, int n, const int64_t *tokens, const int32_t *heads,
                         double *o_rows, double *lse_rows, int n_threads)
{
    if (check_segments(n_seq, cu_q, cu_k, causal) || H < 1 || D < 1) return -1;
    for (int r = 0; r < n; ++r)
        if (tokens[r] < 0 || tokens[r] >= cu_q[n_seq] || heads[r] < 0 || heads[r] >= H) return -1;
    set_threads(n_threads);
    const int Lk_max = max_len(n_seq, cu_k);
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Lk_max > 0 ? Lk_max : 1));
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n; ++r)
            fwd_one(n_seq, cu_q, cu_k, H, D, q, k, v, scale, causal, tokens[r], heads[r],
                    o_rows + (int64_t)r * D, lse_rows + r, s);
        free(s);
    }
    return 0;
}

/*
 * Per-row backward statistics of one (query token, head): m, l and
 * c = sum_j P_j dP_j, and optionally that row's dq.
 */
static void bwd_row(int n_seq, const int32_t *cu_q, const int32_t *cu_k, int H, int D,
                    const double *q, const double *k, const double *v, const double *dO,
                    double scale, int causal, int64_t t, int h, double *m_out, double *l_out,
                    double *c_out, double *dq_row, double *s)
{
    const int b = segment_of(n_seq, cu_q, t);
    const int i = (int)(t - cu_q[b]);
    const int Lk = cu_k[b + 1] - cu_k[b];
    const int nj = admitted(i, Lk, causal);
    const int64_t ld = (int64_t)H * D;
    const double *qi = q + t * ld + (int64_t)h * D;
    const double *dOi = dO + t * ld + (int64_t)h * D;
    const double *k0 = k + (int64_t)cu_k[b] * ld + (int64_t)h * D;
    const double *v0 = v + (int64_t)cu_k[b] * ld + (int64_t)h * D;

    if (dq_row)
        for (int d = 0; d < D; ++d) dq_row[d] = 0.0;
    if (nj == 0) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        *c_out = 0.0;
        return;
    }
    double m, l;
    row_scores(qi, k0, ld, nj, D, scale, s, &m, &l);
    double c = 0.0;
    for (int j = 0; j < nj; ++j) {
        const double p = exp(s[j] - m) / l;
        c += p * dot(dOi, v0 + (int64_t)j * ld, D);
    }
    if (dq_row) {
        for (int j = 0; j < nj; ++j) {
            const double p = exp(s[j] - m) / l;
            const double *kj = k0 + (int64_t)j * ld;
            const double ds = p * (dot(dOi, v0 + (int64_t)j * ld, D) - c);
            for (int d = 0; d < D; ++d) dq_row[d] += scale * ds * kj[d];
        }
    }
    *m_out = m;
    *l_out = l;
    *c_out = c;
}

/*
 * dk and dv of one (key token, head), given the statistics (m, l, c) of every
 * query row of that head (arrays indexed (H, T_q)).
 */
static void bwd_key(int n_seq, const int32_t *cu_q, const int32_t *cu_k, int H, int D,
                    const double *q, const double *k, const double *v, const double *dO,
                    double scale, int causal, int64_t u, int h, const double *m_st,
                    const double *l_st, const double *c_st, double *dk_row, double *dv_row)
{
    const int b = segment_of(n_seq, cu_k, u);
    const int j = (int)(u - cu_k[b]);
    const int Lq = cu_q[b + 1] - cu_q[b];
    const int64_t Tq = cu_q[n_seq];
    const int64_t ld = (int64_t)H * D;
    const double *kj = k + u * ld + (int64_t)h * D;
    const double *vj = v + u * ld + (int64_t)h * D;

    for (int d = 0; d < D; ++d) {
        dk_row[d] = 0.0;
        dv_row[d] = 0.0;
    }
    for (int i = 0; i < Lq; ++i) {
        if (causal && j > i) continue; /* (i, j) not in the relation */
        const int64_t t = cu_q[b] + i;
        const double *qi = q + t * ld + (int64_t)h * D;
        const double *dOi = dO + t * ld + (int64_t)h * D;
        const int64_t st = (int64_t)h * Tq + t;
        const double p = exp(scale * dot(qi, kj, D) - m_st[st]) / l_st[st];
        const double ds = p * (dot(dOi, vj, D) - c_st[st]);
        for (int d = 0; d < D; ++d) {
            dk_row[d] += scale * ds * qi[d];
            dv_row[d] += p * dOi[d];
        }
    }
}

/*
 * Backward.  Computes dq for the listed query rows and dk, dv for the listed
 * key rows.  A NULL token list means "every row" and then the output arrays
 * are full (T, H, D) tensors; otherwise they are (n, D).
 */
int oracle_attn_bwd(int n_seq, const int32_t *cu_q, const int32_t *cu_k, int H, int D,
                    const double *q, const double *k, const double *v, const double *dO,
                    double scale, int causal,
                    int n_q_sel, const int64_t *q_tokens, const int32_t *q_heads, double *dq,
                    int n_k_sel, const int64_t *k_tokens, const int32_t *k_heads, double *dk,
                    double *dv, int n_threads)
{
    if (check_segments(n_seq, cu_q, cu_k, causal) || H < 1 || D < 1) return -1;
    set_threads(n_threads);
    const int64_t Tq = cu_q[n_seq];
    const int64_t Tk = cu_k[n_seq];
    const int Lk_max = max_len(n_seq, cu_k);
    const int64_t nq = q_tokens ? n_q_sel : Tq * H;
    const int64_t nk = k_tokens ? n_k_sel : Tk * H;
    if (q_tokens)
        for (int64_t r = 0; r < nq; ++r)
            if (q_tokens[r] < 0 || q_tokens[r] >= Tq || q_heads[r] < 0 || q_heads[r] >= H) return -1;
    if (k_tokens)
        for (int64_t r = 0; r < nk; ++r)
            if (k_tokens[r] < 0 || k_tokens[r] >= Tk || k_heads[r] < 0 || k_heads[r] >= H) return -1;

    /* Which (segment, head) pairs need the statistics of all their rows. */
    const int64_t n_pairs = (int64_t)n_seq * H;
    unsigned char *need = (unsigned char *)calloc((size_t)n_pairs, 1);
    double *m_st = (double *)malloc(sizeof(double) * (size_t)(Tq * H + 1));
    double *l_st = (double *)malloc(sizeof(double) * (size_t)(Tq * H + 1));
    double *c_st = (double *)malloc(sizeof(double) * (size_t)(Tq * H + 1));
    if (!need || !m_st || !l_st || !c_st) {
        free(need); free(m_st); free(l_st); free(c_st);
        return -2;
    }
    for (int64_t r = 0; r < nk; ++r) {
        const int64_t u = k_tokens ? k_tokens[r] : r / H;
        const int h = k_tokens ? k_heads[r] : (int)(r % H);
        need[(int64_t)segment_of(n_seq, cu_k, u) * H + h] = 1;
    }

    /* Pass 1: statistics of every query row of the needed pairs, and dq. */
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Lk_max > 0 ? Lk_max : 1));
        double m, l, c;
#pragma omp for schedule(dynamic, 8)
        for (int64_t r = 0; r < Tq * H; ++r) {
            const int64_t t = r / H;
            const int h = (int)(r % H);
            if (!need[(int64_t)segment_of(n_seq, cu_q, t) * H + h]) continue;
            bwd_row(n_seq, cu_q, cu_k, H, D, q, k, v, dO, scale, causal, t, h, &m, &l, &c,
                    NULL, s);
            m_st[(int64_t)h * Tq + t] = m;
            l_st[(int64_t)h * Tq + t] = l;
            c_st[(int64_t)h * Tq + t] = c;
        }
#pragma omp for schedule(dynamic, 8)
        for (int64_t r = 0; r < nq; ++r) {
            const int64_t t = q_tokens ? q_tokens[r] : r / H;
            const int h = q_tokens ? q_heads[r] : (int)(r % H);
            bwd_row(n_seq, cu_q, cu_k, H, D, q, k, v, dO, scale, causal, t, h, &m, &l, &c,
                    dq + r * D, s);
        }
        free(s);
    }

    /* Pass 2: dk and dv of the requested keys, one key row at a time. */
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t r = 0; r < nk; ++r) {
        const int64_t u = k_tokens ? k_tokens[r] : r / H;
        const int h = k_tokens ? k_heads[r] : (int)(r % H);
        bwd_key(n_seq, cu_q, cu_k, H, D, q, k, v, dO, scale, causal, u, h, m_st, l_st, c_st,
                dk + r * D, dv + r * D);
    }

    free(need);
    free(m_st);
    free(l_st);
    free(c_st);
    return 0;
}

/*
 * Merge of C partial results (see the header comment): o_parts is (C, T, H, D),
 * lse_parts is (C, H, T), o is (T, H, D), lse is (H, T).  Returns 0, or -1 on
 * bad sizes.
 */
int oracle_attn_merge(int C, int64_t T, int H, int D, const double *o_parts,
                      const double *lse_parts, double *o, double *lse, int n_threads)
{
    if (C < 1 || T < 0 || H < 1 || D < 1) return -1;
    set_threads(n_threads);
    const int64_t n_rows = T * H;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t t = r / H;
        const int h = (int)(r % H);
        double M = -INFINITY;
        for (int c = 0; c < C; ++c) {
            const double x = lse_parts[((int64_t)c * H + h) * T + t];
            if (x > M) M = x;
        }
        double *orow = o + r * D;
        for (int d = 0; d < D; ++d) orow[d] = 0.0;
        if (M == -INFINITY) {
            lse[(int64_t)h * T + t] = -INFINITY;
            continue;
        }
        double l = 0.0;
        for (int c = 0; c < C; ++c) l += exp(lse_parts[((int64_t)c * H + h) * T + t] - M);
        for (int c = 0; c < C; ++c) {
            const double w = exp(lse_parts[((int64_t)c * H + h) * T + t] - M) / l;
            const double *prow = o_parts + ((int64_t)c * T * H + r) * D;
            for (int d = 0; d < D; ++d) orow[d] += w * prow[d];
        }
        lse[(int64_t)h * T + t] = M + log(l);
    }
    return 0;
}

/*
 * Tile-pruned approximate forward (see the header comment): one sequence,
 * full relation.  o is (T_q, H, D), lse is (H, T_q).  n_pruned (optional)
 * receives the number of pruned (query block, key tile) pairs over all heads;
 * min_margin (optional) the smallest |m_tile - (m_run + ln rho)| over all
 * decisions taken against a finite m_run, so that callers can tell whether
 * rounding could flip a decision.  Returns 0, or -1 on bad sizes.
 */
int oracle_attn_fwd_pruned(int64_t Tq, int64_t Tk, int H, int D, const double *q,
                           const double *k, const double *v, double scale, double rho,
                           int block_q, int block_k, double *o, double *lse,
                           int64_t *n_pruned, double *min_margin, int n_threads)
{
    if (Tq < 0 || Tk < 0 || H < 1 || D < 1 || block_q < 1 || block_k < 1) return -1;
    if (!(rho > 0.0 && rho <= 1.0)) return -1;
    set_threads(n_threads);
    const int64_t ld = (int64_t)H * D;
    const int64_t n_qb = (Tq + block_q - 1) / block_q, n_kt = (Tk + block_k - 1) / block_k;
    const double log_rho = log(rho);
    int64_t pruned_total = 0;
    double margin_min = INFINITY;
#pragma omp parallel reduction(+ : pruned_total) reduction(min : margin_min)
    {
        unsigned char *admit = (unsigned char *)malloc((size_t)(n_kt > 0 ? n_kt : 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t blk = 0; blk < n_qb * H; ++blk) {
            const int h = (int)(blk / n_qb);
            const int64_t i0 = (blk % n_qb) * block_q;
            const int64_t i1 = i0 + block_q < Tq ? i0 + block_q : Tq;
            /* decisions: scan the key tiles in order with the block's rolling max */
            double m_run = -INFINITY;
            for (int64_t kt = 0; kt < n_kt; ++kt) {
                const int64_t j0 = kt * block_k, j1 = j0 + block_k < Tk ? j0 + block_k : Tk;
                double m_tile = -INFINITY;
                for (int64_t i = i0; i < i1; ++i)
                    for (int64_t j = j0; j < j1; ++j) {
                        const double x = scale * dot(q + i * ld + (int64_t)h * D,
                                                     k + j * ld + (int64_t)h * D, D);
                        if (x > m_tile) m_tile = x;
                    }
                if (m_run == -INFINITY) {
                    admit[kt] = 1;
                } else {
                    const double margin = m_tile - (m_run + log_rho);
                    admit[kt] = margin >= 0.0;
                    if (fabs(margin) < margin_min) margin_min = fabs(margin);
                }
                if (admit[kt]) {
                    if (m_tile > m_run) m_run = m_tile;
                } else {
                    ++pruned_total;
                }
            }
            /* each row: composed softmax over the keys of the admitted tiles */
            for (int64_t i = i0; i < i1; ++i) {
                const double *qi = q + i * ld + (int64_t)h * D;
                double m = -INFINITY;
                for (int64_t kt = 0; kt < n_kt; ++kt) {
                    if (!admit[kt]) continue;
                    const int64_t j0 = kt * block_k, j1 = j0 + block_k < Tk ? j0 + block_k : Tk;
                    for (int64_t j = j0; j < j1; ++j) {
                        s[j] = scale * dot(qi, k + j * ld + (int64_t)h * D, D);
                        if (s[j] > m) m = s[j];
                    }
                }
                double *orow = o + i * ld + (int64_t)h * D;
                for (int d = 0; d < D; ++d) orow[d] = 0.0;
                if (m == -INFINITY) {
                    lse[(int64_t)h * Tq + i] = -INFINITY;
                    continue;
                }
                double l = 0.0;
                for (int64_t kt = 0; kt < n_kt; ++kt) {
                    if (!admit[kt]) continue;
                    const int64_t j0 = kt * block_k, j1 = j0 + block_k < Tk ? j0 + block_k : Tk;
                    for (int64_t j = j0; j < j1; ++j) l += exp(s[j] - m);
                }
                for (int64_t kt = 0; kt < n_kt; ++kt) {
                    if (!admit[kt]) continue;
                    const int64_t j0 = kt * block_k, j1 = j0 + block_k < Tk ? j0 + block_k : Tk;
                    for (int64_t j = j0; j < j1; ++j) {
                        const double p = exp(s[j] - m) / l;
                        const double *vj = v + j * ld + (int64_t)h * D;
                        for (int d = 0; d < D; ++d) orow[d] += p * vj[d];
                    }
                }
                lse[(int64_t)h * Tq + i] = m + log(l);
            }
        }
        free(s);
        free(admit);
    }
    if (n_pruned) *n_pruned = pruned_total;
    if (min_margin) *min_margin = margin_min;
    return 0;
}

/*
 * Attention over a CSR relation (see the header comment).  row_ptr has n_dst+1
 * nondecreasing offsets from 0; col holds row_ptr[n_dst] source indices in
 * [0, n_src).  scores is (E, H) or NULL (then scores are scale * <q_i, k_j>,
 * q (n_dst, H, D), k (n_src, H, D)).  v is (n_src, H, D); o is (n_dst, H, D),
 * lse (H, n_dst).  Returns 0, or -1 on a malformed relation.
 */
int oracle_csr_fwd(int64_t n_dst, int64_t n_src, const int64_t *row_ptr, const int32_t *col,
                   int H, int D, const double *scores, const double *q, const double *k,
                   const double *v, double scale, double *o, double *lse, int n_threads)
{
    if (n_dst < 0 || n_src < 0 || H < 1 || D < 1 || !row_ptr || row_ptr[0] != 0) return -1;
    for (int64_t i = 0; i < n_dst; ++i)
        if (row_ptr[i + 1] < row_ptr[i]) return -1;
    const int64_t E = row_ptr[n_dst];
    for (int64_t e = 0; e < E; ++e)
        if (col[e] < 0 || col[e] >= n_src) return -1;
    if (!scores && (!q || !k)) return -1;
    set_threads(n_threads);
    const int64_t ld = (int64_t)H * D;
    int64_t max_deg = 0;
    for (int64_t i = 0; i < n_dst; ++i)
        if (row_ptr[i + 1] - row_ptr[i] > max_deg) max_deg = row_ptr[i + 1] - row_ptr[i];
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(max_deg > 0 ? max_deg : 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < n_dst * H; ++r) {
            const int64_t i = r / H;
            const int h = (int)(r % H);
            const int64_t e0 = row_ptr[i], deg = row_ptr[i + 1] - e0;
            double *orow = o + i * ld + (int64_t)h * D;
            for (int d = 0; d < D; ++d) orow[d] = 0.0;
            if (deg == 0) {
                lse[(int64_t)h * n_dst + i] = -INFINITY;
                continue;
            }
            double m = -INFINITY;
            for (int64_t t = 0; t < deg; ++t) {
                const int64_t j = col[e0 + t];
                s[t] = scores ? scores[(e0 + t) * H + h]
                              : scale * dot(q + i * ld + (int64_t)h * D, k + j * ld + (int64_t)h * D, D);
                if (s[t] > m) m = s[t];
            }
            double l = 0.0;
            for (int64_t t = 0; t < deg; ++t) l += exp(s[t] - m);
            for (int64_t t = 0; t < deg; ++t) {
                const double p = exp(s[t] - m) / l;
                const double *vj = v + (int64_t)col[e0 + t] * ld + (int64_t)h * D;
                for (int d = 0; d < D; ++d) orow[d] += p * vj[d];
            }
            lse[(int64_t)h * n_dst + i] = m + log(l);
        }
        free(s);
    }
    return 0;
}
