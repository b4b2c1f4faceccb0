/*
 * oracle.c -- plain, slow, fp64 CPU oracle for online token-eviction
 * compaction of a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or helper with
 * the CUDA library: it is an independent restatement of what the method
 * computes, written for a reader to check against the pages by eye.
 *
 * Sources (web pages on online KV-cache compaction):
 *  [TE]   "Practical Online KV Cache Compaction for LLM Agents: An Empirical
 *         Study" (tutorial page), section "design space: algorithm families
 *         and proxy-query sources", the token-eviction score equation
 *         s_j(Q,K) = ((1/q) * sum_i alpha_ij^2)^(1/2) and the top-m rule
 *         (the raw Key/Value of the m best positions are kept unmodified).
 *  [ACT]  "ActKV 解剖" (zhichai.net analysis of ActKV), the paragraph on the
 *         third component (system engineering): alpha recovered as
 *         exp(logits - LSE); a conflict-free slot plan in which the last X
 *         logical blocks are the target region, retained entries outside it
 *         are paired one-to-one with holes inside it, one parallel copy runs,
 *         and the emptied blocks return to the scheduler.
 *  [SE]   "AI智能体记忆越用越长，推理引擎为何跟不上" (SparseEngine article),
 *         Chain Cache section: the logical prefix is kept apart from physical
 *         storage, so logical positions survive physical deletion.
 *
 * Readings where the pages are silent (each is a fixed choice, tested):
 *  - softmax domain = the n positions of the compacted segment;
 *  - all q*g proxy rows of a GQA group form Q for their KV head;
 *  - ties in the score go to the lower position; keep sets are emitted in
 *    ascending position order;
 *  - X = ceil(m/P); the k-th retained entry outside the target region (in
 *    ascending position) fills the k-th hole of the target region (in
 *    ascending slot order); holes left over are dead (tag -1), their bytes
 *    untouched; the first nb - X blocks of the segment are freed in
 *    ascending block order, sequences in ascending order, pushed onto the
 *    free stack; later block-table entries shift down and vacated entries
 *    become -1.
 *
 * Everything is fp64 (bf16 inputs widen exactly).  No blocking, no fusion.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_NONFINITE (-2)
#define ORC_ERR_NOMEM (-3)
#define ORC_ERR_LAYOUT (-4)
#define ORC_ERR_STACK (-5)

/* bf16 bit pattern -> double (exact widening). */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* ------------------------------------------------------------------------ */
/* Budget (how many positions a unit keeps).                                 */
/* ------------------------------------------------------------------------ */

/* Ratio budget: m = min(n, ceil(ratio * n)).  The 1e-9*n guard keeps products
 * such as 0.07*100 = 7.000000000000001 from rounding up to 8.  A keep ratio
 * of 0.2 (drop 80%) is the setting of the online-compaction study [TE]. */
int64_t oracle_budget_ratio(int64_t n, double ratio)
{
    if (n <= 0) return 0;
    double x = ratio * (double)n - 1e-9 * (double)n;
    int64_t m = (int64_t)ceil(x);
    if (m < 0) m = 0;
    if (m > n) m = n;
    return m;
}

/* ActKV's ratchet budget: start at 512 entries, grow by 1.75x per step,
 * capped at 30 000 entries ([ACT], budget paragraph).  Integer entry count =
 * floor of the product. */
int64_t oracle_budget_actkv(int k)
{
    if (k < 0) return -1;
    double b = 512.0;
    for (int i = 0; i < k; ++i) b *= 1.75;
    double f = floor(b);
    if (f > 30000.0) f = 30000.0;
    return (int64_t)f;
}

/* ------------------------------------------------------------------------ */
/* Scores.                                                                   */
/* ------------------------------------------------------------------------ */

/* One unit, dense fp64 operands.
 *   Q: R x d proxy rows, K: n x d keys (row-major), scale: logit scale.
 *   logits L_ij = scale * sum_t Q_it K_jt
 *   LSE_i = max_j L_ij + log sum_j exp(L_ij - max_j L_ij)      [ACT]
 *   alpha_ij = exp(L_ij - LSE_i)                                [ACT]
 *   s_j = sqrt((1/R) * sum_i alpha_ij^2)                        [TE]
 * Writes s[n] and, if lse != NULL, lse[R]. */
int oracle_score_dense(const double *Q, const double *K, int R, int n, int d,
                       double scale, double *s, double *lse)
{
    if (R <= 0 || n < 0 || d <= 0 || !Q || (n > 0 && (!K || !s))) return ORC_ERR_ARG;
    if (n == 0) {
        if (lse)
            for (int i = 0; i < R; ++i) lse[i] = -INFINITY;
        return ORC_OK;
    }
    double *row = (double *)malloc((size_t)n * sizeof(double));
    if (!row) return ORC_ERR_NOMEM;
    for (int j = 0; j < n; ++j) s[j] = 0.0;

    int status = ORC_OK;
    for (int i = 0; i < R && status == ORC_OK; ++i) {
        const double *qi = Q + (size_t)i * d;
        /* full logit row */
        for (int j = 0; j < n; ++j) {
            const double *kj = K + (size_t)j * d;
            double dot = 0.0;
            for (int t = 0; t < d; ++t) dot += qi[t] * kj[t];
            row[j] = scale * dot;
            if (!isfinite(row[j])) status = ORC_ERR_NONFINITE;
        }
        if (status != ORC_OK) break;
        /* log-sum-exp of the row */
        double mx = row[0];
        for (int j = 1; j < n; ++j)
            if (row[j] > mx) mx = row[j];
        double sum = 0.0;
        for (int j = 0; j < n; ++j) sum += exp(row[j] - mx);
        double lse_i = mx + log(sum);
        if (lse) lse[i] = lse_i;
        /* alpha and its square, accumulated per key */
        for (int j = 0; j < n; ++j) {
            double a = exp(row[j] - lse_i);
            s[j] += a * a;
        }
    }
    if (status == ORC_OK)
        for (int j = 0; j < n; ++j) s[j] = sqrt(s[j] / (double)R);
    free(row);
    return status;
}

/* Action attention of every key (ActKV analysis page, first component: the
 * attention that all action tokens pay to a KV entry, gathered per entry):
 *   a_j = sum_i alpha_ij,  alpha_ij = exp(L_ij - LSE_i) as in
 *   oracle_score_dense; the rows of Q are the action tokens' queries.
 * Writes a[n] and, if lse != NULL, lse[R]. */
int oracle_action_dense(const double *Q, const double *K, int R, int n, int d, double scale,
                        double *a, double *lse)
{
    if (R <= 0 || n < 0 || d <= 0 || !Q || (n > 0 && (!K || !a))) return ORC_ERR_ARG;
    if (n == 0) {
        if (lse)
            for (int i = 0; i < R; ++i) lse[i] = -INFINITY;
        return ORC_OK;
    }
    double *row = (double *)malloc((size_t)n * sizeof(double));
    if (!row) return ORC_ERR_NOMEM;
    for (int j = 0; j < n; ++j) a[j] = 0.0;
    int status = ORC_OK;
    for (int i = 0; i < R && status == ORC_OK; ++i) {
        const double *qi = Q + (size_t)i * d;
        for (int j = 0; j < n; ++j) {
            const double *kj = K + (size_t)j * d;
            double dot = 0.0;
            for (int t = 0; t < d; ++t) dot += qi[t] * kj[t];
            row[j] = scale * dot;
            if (!isfinite(row[j])) status = ORC_ERR_NONFINITE;
        }
        if (status != ORC_OK) break;
        double mx = row[0];
        for (int j = 1; j < n; ++j)
            if (row[j] > mx) mx = row[j];
        double sum = 0.0;
        for (int j = 0; j < n; ++j) sum += exp(row[j] - mx);
        double lse_i = mx + log(sum);
        if (lse) lse[i] = lse_i;
        for (int j = 0; j < n; ++j) a[j] += exp(row[j] - lse_i);
    }
    free(row);
    return status;
}

/* Slot s of sequence b, layer l, head h -> index of its first element in a
 * pool laid out [L][num_pages][H][P][d]. */
static size_t pool_elem(const int32_t *bt_row, int slot, int layer, int head,
                        int num_pages, int H, int P, int d)
{
    int page = bt_row[slot / P];
    int off = slot % P;
    return ((((size_t)layer * num_pages + (size_t)page) * H + head) * P + off) * (size_t)d;
}

static size_t tag_elem(const int32_t *bt_row, int slot, int layer, int head,
                       int num_pages, int H, int P)
{
    int page = bt_row[slot / P];
    int off = slot % P;
    return (((size_t)layer * num_pages + (size_t)page) * H + head) * P + off;
}

/* Checks one sequence's segment against the layout rules: the segment starts
 * on a block boundary and ends on one unless it ends the sequence; every
 * block it touches is mapped to a valid page. */
static int check_segment(const int32_t *bt_row, int nblocks_b, int max_blocks, int num_pages,
                         int P, int s0, int s1, int seq_len)
{
    if (s0 < 0 || s1 < s0 || s1 > seq_len) return ORC_ERR_LAYOUT;
    if (s0 % P != 0) return ORC_ERR_LAYOUT;
    if (s1 % P != 0 && s1 != seq_len) return ORC_ERR_LAYOUT;
    if (ceil_div(seq_len, P) > nblocks_b || nblocks_b > max_blocks) return ORC_ERR_LAYOUT;
    for (int blk = s0 / P; blk < ceil_div(s1, P); ++blk)
        if (bt_row[blk] < 0 || bt_row[blk] >= num_pages) return ORC_ERR_LAYOUT;
    return ORC_OK;
}

/* Scores of every (sequence b, layer l, KV head h) unit of a paged cache.
 *   k_pool   bf16 bits [L][num_pages][H][P][d]
 *   q        bf16 bits [B][L][H][R][d]  (R = proxy rows of the GQA group)
 *   segments [seg_start[b], seg_end[b]) in the sequence's slot coordinates
 *   unit_mask [B][L][H] (nonzero = compute) or NULL for all units
 *   scores   out [L][H][Ntot], Ntot = sum_b n_b, sequence b at offset
 *            sum_{b'<b} n_b'   (entries of skipped units are left untouched)
 *   lse      out [B][L][H][R] or NULL */
static int cache_units(const uint16_t *k_pool, const int32_t *block_table, const int32_t *nblocks,
                       int max_blocks, int L, int num_pages, int H, int P, int d,
                       const int32_t *seg_start, const int32_t *seg_end, const int32_t *seq_len,
                       int B, const uint16_t *q, int R, double scale, const uint8_t *unit_mask,
                       double *scores, double *lse, int nthreads, int action)
{
    if (!k_pool || !block_table || !nblocks || !seg_start || !seg_end || !seq_len || !q ||
        !scores || L <= 0 || H <= 0 || P <= 0 || d <= 0 || R <= 0 || B <= 0)
        return ORC_ERR_ARG;
    int64_t *off = (int64_t *)malloc((size_t)(B + 1) * sizeof(int64_t));
    if (!off) return ORC_ERR_NOMEM;
    off[0] = 0;
    for (int b = 0; b < B; ++b) {
        int st = check_segment(block_table + (size_t)b * max_blocks, nblocks[b], max_blocks,
                               num_pages, P, seg_start[b], seg_end[b], seq_len[b]);
        if (st != ORC_OK) {
            free(off);
            return st;
        }
        off[b + 1] = off[b] + (seg_end[b] - seg_start[b]);
    }
    const int64_t Ntot = off[B];
    const int64_t units = (int64_t)B * L * H;
    int status = ORC_OK;
    if (nthreads <= 0) nthreads = 1;

#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t u = 0; u < units; ++u) {
        int b = (int)(u / ((int64_t)L * H));
        int l = (int)((u / H) % L);
        int h = (int)(u % H);
        if (unit_mask && !unit_mask[u]) continue;
        int s0 = seg_start[b], n = seg_end[b] - seg_start[b];
        const int32_t *bt_row = block_table + (size_t)b * max_blocks;
        double *Qd = (double *)malloc((size_t)R * d * sizeof(double));
        double *Kd = (double *)malloc(((size_t)(n > 0 ? n : 1)) * d * sizeof(double));
        double *lse_u = lse ? lse + (size_t)u * R : NULL;
        if (!Qd || !Kd) {
#pragma omp critical
            status = ORC_ERR_NOMEM;
            free(Qd);
            free(Kd);
            continue;
        }
        const uint16_t *qu = q + (size_t)u * R * d; /* [B][L][H] == unit order */
        for (size_t e = 0; e < (size_t)R * d; ++e) Qd[e] = bf16_to_double(qu[e]);
        /* gather the unit's keys through the block table */
        for (int j = 0; j < n; ++j) {
            size_t base = pool_elem(bt_row, s0 + j, l, h, num_pages, H, P, d);
            for (int t = 0; t < d; ++t) Kd[(size_t)j * d + t] = bf16_to_double(k_pool[base + t]);
        }
        double *s_u = scores + ((size_t)l * H + h) * Ntot + off[b];
        int st = action ? oracle_action_dense(Qd, Kd, R, n, d, scale, s_u, lse_u)
                        : oracle_score_dense(Qd, Kd, R, n, d, scale, s_u, lse_u);
        if (st != ORC_OK) {
#pragma omp critical
            status = st;
        }
        free(Qd);
        free(Kd);
    }
    free(off);
    return status;
}

int oracle_score_cache(const uint16_t *k_pool, const int32_t *block_table, const int32_t *nblocks,
                       int max_blocks, int L, int num_pages, int H, int P, int d,
                       const int32_t *seg_start, const int32_t *seg_end, const int32_t *seq_len,
                       int B, const uint16_t *q, int R, double scale, const uint8_t *unit_mask,
                       double *scores, double *lse, int nthreads)
{
    return cache_units(k_pool, block_table, nblocks, max_blocks, L, num_pages, H, P, d, seg_start,
                       seg_end, seq_len, B, q, R, scale, unit_mask, scores, lse, nthreads, 0);
}

/* Action attention a_j (oracle_action_dense) of every unit of a paged cache,
 * laid out like oracle_score_cache's scores. */
int oracle_action_cache(const uint16_t *k_pool, const int32_t *block_table, const int32_t *nblocks,
                        int max_blocks, int L, int num_pages, int H, int P, int d,
                        const int32_t *seg_start, const int32_t *seg_end, const int32_t *seq_len,
                        int B, const uint16_t *q, int R, double scale, const uint8_t *unit_mask,
                        double *a, double *lse, int nthreads)
{
    return cache_units(k_pool, block_table, nblocks, max_blocks, L, num_pages, H, P, d, seg_start,
                       seg_end, seq_len, B, q, R, scale, unit_mask, a, lse, nthreads, 1);
}

/* ------------------------------------------------------------------------ */
/* Top-m selection.                                                          */
/* ------------------------------------------------------------------------ */

typedef struct {
    double s;
    int32_t j;
} scored_pos;

/* higher score first; equal scores -> lower position first */
static int by_score_then_position(const void *pa, const void *pb)
{
    const scored_pos *a = (const scored_pos *)pa, *b = (const scored_pos *)pb;
    if (a->s > b->s) return -1;
    if (a->s < b->s) return 1;
    return (a->j > b->j) - (a->j < b->j);
}

static int ascending_int(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/* Keep the m positions with the highest s_j [TE]; ties -> lower j; emitted
 * in ascending position order.  m > n keeps everything.  Returns the number
 * kept, or a negative error. */
int oracle_select(const double *s, int n, int m, int32_t *keep)
{
    if (n < 0 || m < 0 || (n > 0 && !s)) return ORC_ERR_ARG;
    if (m > n) m = n;
    if (m == 0) return 0;
    if (!keep) return ORC_ERR_ARG;
    scored_pos *e = (scored_pos *)malloc((size_t)n * sizeof(scored_pos));
    if (!e) return ORC_ERR_NOMEM;
    for (int j = 0; j < n; ++j) {
        if (!isfinite(s[j])) {
            free(e);
            return ORC_ERR_NONFINITE;
        }
        e[j].s = s[j];
        e[j].j = j;
    }
    qsort(e, (size_t)n, sizeof(scored_pos), by_score_then_position);
    for (int r = 0; r < m; ++r) keep[r] = e[r].j;
    qsort(keep, (size_t)m, sizeof(int32_t), ascending_int);
    free(e);
    return m;
}

/* Selection for every unit.  scores [L][H][Ntot] as produced above, m[b] the
 * budget of sequence b (clamped to n_b), keep out [L][H][Mtot] with sequence
 * b at offset sum_{b'<b} min(m_b', n_b'). */
int oracle_select_cache(const double *scores, int L, int H, const int32_t *seg_start,
                        const int32_t *seg_end, int B, const int32_t *m, int32_t *keep,
                        int nthreads)
{
    if (!scores || !seg_start || !seg_end || !m || !keep || L <= 0 || H <= 0 || B <= 0)
        return ORC_ERR_ARG;
    int64_t Ntot = 0, Mtot = 0;
    for (int b = 0; b < B; ++b) {
        int n = seg_end[b] - seg_start[b];
        if (n < 0 || m[b] < 0) return ORC_ERR_ARG;
        Ntot += n;
        Mtot += (m[b] < n ? m[b] : n);
    }
    int status = ORC_OK;
    if (nthreads <= 0) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t lh = 0; lh < (int64_t)L * H; ++lh) {
        int64_t noff = 0, moff = 0;
        for (int b = 0; b < B; ++b) {
            int n = seg_end[b] - seg_start[b];
            int mb = m[b] < n ? m[b] : n;
            int got = oracle_select(scores + lh * Ntot + noff, n, mb, keep + lh * Mtot + moff);
            if (got != mb) {
#pragma omp critical
                status = got < 0 ? got : ORC_ERR_ARG;
            }
            noff += n;
            moff += mb;
        }
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Compaction: naive sequential simulation of the slot plan [ACT].           */
/* ------------------------------------------------------------------------ */

/* Moves the retained entries of every unit of the layers held in the given
 * pool slices (layer_lo .. layer_lo+Lpart-1 of the cache; the slices hold
 * only those layers, each [Lpart][num_pages][H][P][d] / [..][P] for tags).
 * keep [L_total][H][Mtot] as produced by selection; only rows of the held
 * layers are read.
 *
 * For a unit with n positions and budget m: nb = ceil(n/P) blocks, X =
 * ceil(m/P), the target region T is the last X blocks of the segment,
 * i.e. segment slots [Bs, Bs + X*P) with Bs = (nb - X)*P.  Walking T's
 * slots in ascending order, a slot that is not a retained position (evicted,
 * or past the segment end inside the last block) is a hole: it receives the
 * next retained entry that lies before Bs (ascending), K/V bytes and tag,
 * or, when none is left, tag -1 with its bytes untouched.  Retained entries
 * inside T never move. */
int oracle_compact_layers(uint16_t *k_pool, uint16_t *v_pool, int32_t *tags, int layer_lo,
                          int Lpart, int L_total, int num_pages, int H, int P, int d,
                          const int32_t *block_table, int max_blocks, const int32_t *seg_start,
                          const int32_t *seg_end, int B, const int32_t *m, const int32_t *keep)
{
    if (!k_pool || !v_pool || !tags || !block_table || !seg_start || !seg_end || !m || !keep ||
        Lpart <= 0 || layer_lo < 0 || layer_lo + Lpart > L_total || H <= 0 || P <= 0 || d <= 0)
        return ORC_ERR_ARG;
    int64_t Mtot = 0;
    for (int b = 0; b < B; ++b) {
        int n = seg_end[b] - seg_start[b];
        Mtot += (m[b] < n ? m[b] : n);
    }
    for (int lp = 0; lp < Lpart; ++lp) {
        int l = layer_lo + lp;
        for (int h = 0; h < H; ++h) {
            int64_t moff = 0;
            for (int b = 0; b < B; ++b) {
                int s0 = seg_start[b], n = seg_end[b] - seg_start[b];
                int mb = m[b] < n ? m[b] : n;
                const int32_t *ku = keep + ((int64_t)l * H + h) * Mtot + moff;
                moff += mb;
                if (n == 0) continue;
                const int32_t *bt_row = block_table + (size_t)b * max_blocks;
                int nb = (int)ceil_div(n, P), X = (int)ceil_div(mb, P);
                int Bs = (nb - X) * P;
                /* retained flags of the segment */
                uint8_t *kept = (uint8_t *)calloc((size_t)n, 1);
                if (!kept) return ORC_ERR_NOMEM;
                for (int r = 0; r < mb; ++r) {
                    if (ku[r] < 0 || ku[r] >= n || (r > 0 && ku[r] <= ku[r - 1])) {
                        free(kept);
                        return ORC_ERR_ARG;
                    }
                    kept[ku[r]] = 1;
                }
                int cursor = 0; /* next retained entry before Bs */
                for (int t = Bs; t < Bs + X * P; ++t) {
                    if (t < n && kept[t]) continue;          /* survivor in T: stays */
                    size_t dt = tag_elem(bt_row, s0 + t, lp, h, num_pages, H, P);
                    if (cursor < mb && ku[cursor] < Bs) {   /* hole: fill it */
                        int src = ku[cursor++];
                        size_t se = pool_elem(bt_row, s0 + src, lp, h, num_pages, H, P, d);
                        size_t de = pool_elem(bt_row, s0 + t, lp, h, num_pages, H, P, d);
                        memcpy(k_pool + de, k_pool + se, (size_t)d * sizeof(uint16_t));
                        memcpy(v_pool + de, v_pool + se, (size_t)d * sizeof(uint16_t));
                        tags[dt] = tags[tag_elem(bt_row, s0 + src, lp, h, num_pages, H, P)];
                    } else {                                  /* hole left dead */
                        tags[dt] = -1;
                    }
                }
                free(kept);
            }
        }
    }
    return ORC_OK;
}

/* Returns the emptied blocks to the allocator [ACT]: for each sequence in
 * ascending order, the first nb - X blocks of its segment are pushed, in
 * ascending block order, onto the free stack (free_ids[(*free_top)++]);
 * they leave the block table, later entries shift down, the vacated tail
 * entries become -1, and nblocks[b] drops by nb - X.  Logical positions are
 * untouched (they live in the tags) [SE]. */
int oracle_free_blocks(int32_t *block_table, int32_t *nblocks, int max_blocks, int32_t *free_ids,
                       int32_t *free_top, int capacity, int P, const int32_t *seg_start,
                       const int32_t *seg_end, int B, const int32_t *m)
{
    if (!block_table || !nblocks || !free_ids || !free_top || !seg_start || !seg_end || !m ||
        P <= 0 || B <= 0)
        return ORC_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        int n = seg_end[b] - seg_start[b];
        if (n == 0) continue;
        int mb = m[b] < n ? m[b] : n;
        int nb = (int)ceil_div(n, P), X = (int)ceil_div(mb, P);
        int f = nb - X, sb = seg_start[b] / P;
        int32_t *row = block_table + (size_t)b * max_blocks;
        if (*free_top + f > capacity) return ORC_ERR_STACK;
        for (int i = 0; i < f; ++i) free_ids[(*free_top)++] = row[sb + i];
        int old = nblocks[b];
        for (int i = sb; i < old - f; ++i) row[i] = row[i + f];
        for (int i = old - f; i < old; ++i) row[i] = -1;
        nblocks[b] = old - f;
    }
    return ORC_OK;
}

/* Order-preserving, out-of-place logical view of one unit [TE][SE]: the
 * r-th retained position's K bytes, V bytes and logical position (its tag
 * before compaction), r = 0..m-1 in ascending position order. */
int oracle_logical_view(const uint16_t *k_pool, const uint16_t *v_pool, const int32_t *tags,
                        int layer, int head, int num_pages, int H, int P, int d,
                        const int32_t *bt_row, int s0, const int32_t *keep, int m, uint16_t *Kc,
                        uint16_t *Vc, int32_t *pos)
{
    if (!k_pool || !v_pool || !tags || !bt_row || (m > 0 && (!keep || !Kc || !Vc || !pos)))
        return ORC_ERR_ARG;
    for (int r = 0; r < m; ++r) {
        size_t e = pool_elem(bt_row, s0 + keep[r], layer, head, num_pages, H, P, d);
        memcpy(Kc + (size_t)r * d, k_pool + e, (size_t)d * sizeof(uint16_t));
        memcpy(Vc + (size_t)r * d, v_pool + e, (size_t)d * sizeof(uint16_t));
        pos[r] = tags[tag_elem(bt_row, s0 + keep[r], layer, head, num_pages, H, P)];
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Layout-preserving eviction and order-preserving fresh-page compaction.    */
/* ------------------------------------------------------------------------ */

/* bf16 bit pattern nearest to x (round to nearest, ties to even), finite x. */
static uint16_t bf16_bits_nearest(double x)
{
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* The sentinel key element of a dead slot, bf16(-10^4) [IK]. */
uint16_t oracle_sentinel_k_bits(void) { return bf16_bits_nearest(-1.0e4); }

/* Checks a unit's keep list (ascending, inside [0, n)) and marks it. */
static int mark_kept(const int32_t *ku, int mb, int n, uint8_t *kept)
{
    for (int r = 0; r < mb; ++r) {
        if (ku[r] < 0 || ku[r] >= n || (r > 0 && ku[r] <= ku[r - 1])) return ORC_ERR_ARG;
        kept[ku[r]] = 1;
    }
    return ORC_OK;
}

/* Layout-preserving eviction ("IntentKV: Cross-Turn Intent-Aware KV Cache
 * Pruning", section on layout-preserving eviction): an evicted position is
 * turned into a dead slot whose K/V are constants that remove its attention
 * contribution (K = -10^4, V = 0) while every retained entry keeps its
 * physical slot.  Reading: each of the d key elements of an evicted position
 * becomes bf16(-10^4), each value element +0, its tag -1; retained entries,
 * slots past the segment end, the block table and the allocator are left as
 * they are (no page is freed).  Pool slices hold layers
 * [layer_lo, layer_lo + Lpart); keep is [L_total][H][Mtot]. */
int oracle_evict_sentinel(uint16_t *k_pool, uint16_t *v_pool, int32_t *tags, int layer_lo,
                          int Lpart, int L_total, int num_pages, int H, int P, int d,
                          const int32_t *block_table, int max_blocks, const int32_t *seg_start,
                          const int32_t *seg_end, int B, const int32_t *m, const int32_t *keep)
{
    if (!k_pool || !v_pool || !tags || !block_table || !seg_start || !seg_end || !m || !keep ||
        Lpart <= 0 || layer_lo < 0 || layer_lo + Lpart > L_total || H <= 0 || P <= 0 || d <= 0)
        return ORC_ERR_ARG;
    const uint16_t ks = oracle_sentinel_k_bits();
    int64_t Mtot = 0;
    for (int b = 0; b < B; ++b) {
        int n = seg_end[b] - seg_start[b];
        Mtot += (m[b] < n ? m[b] : n);
    }
    for (int lp = 0; lp < Lpart; ++lp) {
        int l = layer_lo + lp;
        for (int h = 0; h < H; ++h) {
            int64_t moff = 0;
            for (int b = 0; b < B; ++b) {
                int s0 = seg_start[b], n = seg_end[b] - seg_start[b];
                int mb = m[b] < n ? m[b] : n;
                const int32_t *ku = keep + ((int64_t)l * H + h) * Mtot + moff;
                moff += mb;
                if (n == 0) continue;
                const int32_t *bt_row = block_table + (size_t)b * max_blocks;
                uint8_t *kept = (uint8_t *)calloc((size_t)n, 1);
                if (!kept) return ORC_ERR_NOMEM;
                if (mark_kept(ku, mb, n, kept) != ORC_OK) {
                    free(kept);
                    return ORC_ERR_ARG;
                }
                for (int t = 0; t < n; ++t) {
                    if (kept[t]) continue;
                    size_t e = pool_elem(bt_row, s0 + t, lp, h, num_pages, H, P, d);
                    for (int c = 0; c < d; ++c) {
                        k_pool[e + c] = ks;
                        v_pool[e + c] = 0;
                    }
                    tags[tag_elem(bt_row, s0 + t, lp, h, num_pages, H, P)] = -1;
                }
                free(kept);
            }
        }
    }
    return ORC_OK;
}

/* Order-preserving compaction into fresh pages (the order objection of the
 * IntentKV page, met by moving survivors instead of renumbering them in
 * place).  Reading: a sequence whose segment keeps fewer than all of its n
 * positions ("active") takes X = ceil(m/P) fresh pages from the free stack;
 * the pops of all active sequences, in ascending sequence order, come before
 * any page is returned.  This function lists them: fresh[k] is the page the
 * k-th pop hands out, free_ids[top - 1 - k].  Writes the count to *count;
 * fails if the stack holds fewer pages. */
int oracle_fresh_pages(const int32_t *free_ids, int32_t free_top, int P, const int32_t *seg_start,
                       const int32_t *seg_end, int B, const int32_t *m, int32_t *fresh,
                       int32_t *count)
{
    if (!free_ids || !seg_start || !seg_end || !m || !count || P <= 0 || B <= 0) return ORC_ERR_ARG;
    int32_t k = 0;
    for (int b = 0; b < B; ++b) {
        int n = seg_end[b] - seg_start[b];
        int mb = m[b] < n ? m[b] : n;
        if (n == 0 || mb == n) continue;
        int X = (int)ceil_div(mb, P);
        for (int x = 0; x < X; ++x, ++k) {
            if (free_top - 1 - k < 0) return ORC_ERR_STACK;
            if (fresh) fresh[k] = free_ids[free_top - 1 - k];
        }
    }
    *count = k;
    return ORC_OK;
}

/* The copy of the fresh-page compaction: in every unit of an active
 * sequence the r-th retained position (ascending) goes to slot r of the
 * sequence's fresh pages (page fresh[xoff + r / P], offset r % P) with its K
 * bytes, V bytes and tag; slots r = m .. X*P-1 of the last fresh page get tag
 * -1, bytes untouched.  Sources are read through the old block table; fresh
 * pages are disjoint from every mapped page, so the order of copies does not
 * matter.  Inactive sequences (m = n) are left alone. */
int oracle_compact_fresh(uint16_t *k_pool, uint16_t *v_pool, int32_t *tags, int layer_lo,
                         int Lpart, int L_total, int num_pages, int H, int P, int d,
                         const int32_t *block_table, int max_blocks, const int32_t *seg_start,
                         const int32_t *seg_end, int B, const int32_t *m, const int32_t *keep,
                         const int32_t *fresh)
{
    if (!k_pool || !v_pool || !tags || !block_table || !seg_start || !seg_end || !m || !keep ||
        !fresh || Lpart <= 0 || layer_lo < 0 || layer_lo + Lpart > L_total || H <= 0 || P <= 0 ||
        d <= 0)
        return ORC_ERR_ARG;
    int64_t Mtot = 0;
    for (int b = 0; b < B; ++b) {
        int n = seg_end[b] - seg_start[b];
        Mtot += (m[b] < n ? m[b] : n);
    }
    for (int lp = 0; lp < Lpart; ++lp) {
        int l = layer_lo + lp;
        for (int h = 0; h < H; ++h) {
            int64_t moff = 0;
            int xoff = 0;
            for (int b = 0; b < B; ++b) {
                int s0 = seg_start[b], n = seg_end[b] - seg_start[b];
                int mb = m[b] < n ? m[b] : n;
                const int32_t *ku = keep + ((int64_t)l * H + h) * Mtot + moff;
                moff += mb;
                if (n == 0 || mb == n) continue;
                int X = (int)ceil_div(mb, P);
                const int32_t *bt_row = block_table + (size_t)b * max_blocks;
                for (int r = 0; r < mb; ++r)
                    if (ku[r] < 0 || ku[r] >= n || (r > 0 && ku[r] <= ku[r - 1])) return ORC_ERR_ARG;
                for (int r = 0; r < X * P; ++r) {
                    int page = fresh[xoff + r / P];
                    size_t dt = (((size_t)lp * num_pages + (size_t)page) * H + h) * P + (size_t)(r % P);
                    if (r < mb) {
                        size_t se = pool_elem(bt_row, s0 + ku[r], lp, h, num_pages, H, P, d);
                        memcpy(k_pool + dt * d, k_pool + se, (size_t)d * sizeof(uint16_t));
                        memcpy(v_pool + dt * d, v_pool + se, (size_t)d * sizeof(uint16_t));
                        tags[dt] = tags[tag_elem(bt_row, s0 + ku[r], lp, h, num_pages, H, P)];
                    } else {
                        tags[dt] = -1;
                    }
                }
                xoff += X;
            }
        }
    }
    return ORC_OK;
}

/* The bookkeeping of the fresh-page compaction: the stack loses the popped
 * pages (top -= sum X), then every active sequence, in ascending order,
 * returns all nb blocks of its old segment in ascending block order; in its
 * block-table row the segment's nb entries are replaced by its X fresh
 * pages, later entries shift down by nb - X, vacated tail entries become -1
 * and nblocks drops by nb - X.  `fresh` is the list of oracle_fresh_pages. */
int oracle_commit_fresh(int32_t *block_table, int32_t *nblocks, int max_blocks, int32_t *free_ids,
                        int32_t *free_top, int capacity, int P, const int32_t *seg_start,
                        const int32_t *seg_end, int B, const int32_t *m, const int32_t *fresh)
{
    if (!block_table || !nblocks || !free_ids || !free_top || !seg_start || !seg_end || !m ||
        P <= 0 || B <= 0)
        return ORC_ERR_ARG;
    int32_t count = 0;
    int st = oracle_fresh_pages(free_ids, *free_top, P, seg_start, seg_end, B, m, NULL, &count);
    if (st != ORC_OK) return st;
    if (count > 0 && !fresh) return ORC_ERR_ARG;
    *free_top -= count;
    int xoff = 0;
    for (int b = 0; b < B; ++b) {
        int n = seg_end[b] - seg_start[b];
        int mb = m[b] < n ? m[b] : n;
        if (n == 0 || mb == n) continue;
        int nb = (int)ceil_div(n, P), X = (int)ceil_div(mb, P), sb = seg_start[b] / P;
        int32_t *row = block_table + (size_t)b * max_blocks;
        if (*free_top + nb > capacity) return ORC_ERR_STACK;
        for (int i = 0; i < nb; ++i) free_ids[(*free_top)++] = row[sb + i];
        int old = nblocks[b], f = nb - X;
        for (int x = 0; x < X; ++x) row[sb + x] = fresh[xoff + x];
        for (int i = sb + X; i < old - f; ++i) row[i] = row[i + f];
        for (int i = old - f; i < old; ++i) row[i] = -1;
        nblocks[b] = old - f;
        xoff += X;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* ActKV action-critical entries and LRFU.                                   */
/* ------------------------------------------------------------------------ */

/* Action-critical entries of one unit (ActKV analysis page, first component:
 * entries whose action attention falls within the top 90% count as action-
 * critical).  Reading: order the entries by a_j (descending, ties to the
 * lower position), take the shortest prefix whose cumulative a reaches
 * frac * sum_j a_j, and mark every entry whose a_j is at least the last
 * value of that prefix (ties at the boundary included).  hit[n] gets 0/1.
 * An all-zero a marks nothing. */
int oracle_action_hits(const double *a, int n, double frac, uint8_t *hit)
{
    if (n < 0 || (n > 0 && (!a || !hit)) || !(frac >= 0.0 && frac <= 1.0)) return ORC_ERR_ARG;
    if (n == 0) return ORC_OK;
    scored_pos *v = (scored_pos *)malloc((size_t)n * sizeof(scored_pos));
    if (!v) return ORC_ERR_NOMEM;
    double total = 0.0;
    for (int j = 0; j < n; ++j) {
        v[j].s = a[j];
        v[j].j = j;
        total += a[j];
        hit[j] = 0;
    }
    if (total > 0.0 && frac > 0.0) {
        qsort(v, (size_t)n, sizeof(scored_pos), by_score_then_position);
        double cum = 0.0, tau = v[n - 1].s;
        for (int r = 0; r < n; ++r) {
            cum += v[r].s;
            if (cum >= frac * total) {
                tau = v[r].s;
                break;
            }
        }
        for (int j = 0; j < n; ++j) hit[j] = (uint8_t)(a[j] >= tau);
    }
    free(v);
    return ORC_OK;
}

/* One LRFU step over every unit of a paged cache (ActKV analysis page: LRFU
 * with its hit signal replaced by "hit by action attention", decay lambda =
 * 0.5).  LRFU's combined recency-frequency value of an entry referenced at
 * times t_k is sum_k (1/2)^(lambda (t - t_k)); evaluated once per compaction
 * step it is  crf <- 2^(-lambda) crf + hit.  crf_pool holds one value per
 * slot [L][num_pages][H][P] and is updated in place for the positions of
 * each segment; crf_out [L][H][Ntot] receives the new values (the eviction
 * scores) and hits [L][H][Ntot] (may be NULL) the hit flags. */
int oracle_lrfu_cache(double *crf_pool, int L, int num_pages, int H, int P,
                      const int32_t *block_table, int max_blocks, const int32_t *seg_start,
                      const int32_t *seg_end, int B, const double *a, double frac, double lambda,
                      double *crf_out, uint8_t *hits)
{
    if (!crf_pool || !block_table || !seg_start || !seg_end || !a || !crf_out || L <= 0 ||
        H <= 0 || P <= 0 || B <= 0)
        return ORC_ERR_ARG;
    int64_t Ntot = 0;
    for (int b = 0; b < B; ++b) Ntot += seg_end[b] - seg_start[b];
    const double decay = pow(2.0, -lambda);
    for (int l = 0; l < L; ++l) {
        for (int h = 0; h < H; ++h) {
            int64_t off = 0;
            for (int b = 0; b < B; ++b) {
                int s0 = seg_start[b], n = seg_end[b] - seg_start[b];
                const size_t row = ((size_t)l * H + h) * (size_t)Ntot + (size_t)off;
                off += n;
                if (n == 0) continue;
                uint8_t *hit = (uint8_t *)malloc((size_t)n);
                if (!hit) return ORC_ERR_NOMEM;
                int st = oracle_action_hits(a + row, n, frac, hit);
                if (st != ORC_OK) {
                    free(hit);
                    return st;
                }
                const int32_t *bt_row = block_table + (size_t)b * max_blocks;
                for (int j = 0; j < n; ++j) {
                    size_t e = tag_elem(bt_row, s0 + j, l, h, num_pages, H, P);
                    crf_pool[e] = decay * crf_pool[e] + (double)hit[j];
                    crf_out[row + j] = crf_pool[e];
                    if (hits) hits[row + j] = hit[j];
                }
                free(hit);
            }
        }
    }
    return ORC_OK;
}
