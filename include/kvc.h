/*
 * kvc.h -- C ABI of libkvc: online token-eviction compaction of a paged KV
 * cache on one GB300 (sm_103a).
 *
 * The five calls below are, in order, the data-parallel hot path:
 *
 *   kvc_score        proxy-query attention-mass score of every cached key
 *   kvc_select_topm  top-m positions per (layer, KV head, sequence)
 *   kvc_plan_compact conflict-free slot plan (tail target region)
 *   kvc_compact      one parallel copy of the retained entries
 *   kvc_free_pages   emptied blocks back to the allocator
 *
 * Sources (web pages on online KV-cache compaction):
 *   [TE]  "Practical Online KV Cache Compaction for LLM Agents: An Empirical
 *         Study" (tutorial page), section on the design space: proxy queries
 *         Q (q x d) give attention weights alpha_ij over the context to be
 *         compacted; s_j(Q,K) = ((1/q) sum_i alpha_ij^2)^(1/2); the top-m
 *         positions keep their raw Key/Value, the rest are dropped; keep
 *         ratio 0.2; delayed (next-turn) queries as proxies.
 *   [ACT] "ActKV 解剖" (zhichai.net analysis of ActKV), paragraph on the third
 *         component: attention recovered as exp(logits - LSE) without the
 *         full attention matrix; a conflict-free slot plan whose target is
 *         the last X logical blocks, retained entries outside it paired
 *         one-to-one with holes inside it, one parallel copy, emptied blocks
 *         returned to the scheduler, no extra KV buffer; budget paragraph:
 *         512 entries, x1.75 per growth step, cap 30 000.
 *   [SE]  "AI智能体记忆越用越长，推理引擎为何跟不上" (SparseEngine article):
 *         the application names a history range and a retain ratio
 *         (controllable prefix-cache pruning); Chain Cache keeps the logical
 *         prefix apart from physical storage.
 *
 * Conventions
 *   Ownership: the caller owns every buffer; the library allocates no device
 *     or pinned memory and keeps no state across calls except the device
 *     status word (kvc_read_device_status) and cached TMA descriptors.
 *   Device reset: the device addresses of the library's own device arrays
 *     (the status word, the kvc_score_noalloc scratch) are looked up once per
 *     device and kept for the life of the process, so resetting a device
 *     (cudaDeviceReset) while the library is loaded is not supported: a call
 *     made after a reset may use a stale address.  Restart the process instead.
 *   Pointers: device pointers unless marked "host".  k_pool, v_pool, q and
 *     workspaces must be 16-byte aligned.
 *   Streams: every call is asynchronous on `stream` (0 = legacy default
 *     stream) and performs no implicit synchronisation.  Calls of one
 *     compaction must be issued in order on the same stream.
 *   Errors: arguments are validated on the host before any launch; a bad
 *     argument returns a negative kvc_status and launches nothing.  The text
 *     of the last error of the calling thread is kvc_last_error().  Errors a
 *     kernel detects (bounded wait expired, free stack overflow, a block-table
 *     entry out of range) set bits of the device status word instead of
 *     trapping.  Checked mode (environment variable KVC_CHECKED set and not
 *     "0"): every call that launched work synchronises its stream and returns
 *     KVC_ERR_DEVICE_CHECK if the status word has a bit set (not while the
 *     stream is being captured into a graph).
 *   Tracing: each call is an NVTX range named after it.
 *   Cache layout (all layers share one block table and one page id space):
 *     k_pool, v_pool  bf16  [L][num_pages][H][P][d]  (H = KV heads)
 *     tags            int32 [L][num_pages][H][P]     logical position of the
 *                     entry in the slot, -1 = empty/dead ([SE] Chain Cache)
 *     block_table     int32 [B][max_blocks], nblocks int32 [B]
 *   Slot coordinates: slot s of sequence b lives in page
 *     block_table[b][s / P] at offset s % P.  A segment is a slot range
 *     [seg_start, seg_end) of one sequence: seg_start % P == 0 and
 *     (seg_end % P == 0 or seg_end == seq_len[b]).
 *   Supported: d in {64, 128}; P a power of two in [8, 64]; 1 <= R <= 4096;
 *     L*num_pages*H*P < 2^31.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t kvc_status;
#define KVC_OK 0
#define KVC_ERR_INVALID_ARG (-1)       /* null pointer, bad size or alignment   */
#define KVC_ERR_UNALIGNED_SEGMENT (-2) /* segment not on block boundaries       */
#define KVC_ERR_BUDGET (-3)            /* m < 0                                 */
#define KVC_ERR_WORKSPACE (-4)         /* workspace or plan buffer too small    */
#define KVC_ERR_UNSUPPORTED (-5)       /* d, P or R outside the supported set   */
#define KVC_ERR_CUDA (-6)              /* CUDA runtime/driver error             */
#define KVC_ERR_DEVICE_CHECK (-7)      /* checked mode: status word has a bit set */

/* Device status word bits (kvc_read_device_status). */
#define KVC_DEV_WAIT_TIMEOUT 1u /* a bounded pipeline wait gave up           */
#define KVC_DEV_FREE_STACK 2u   /* free stack too full (push) or too empty (fresh-page pop) */
#define KVC_DEV_BAD_PAGE 4u     /* a block-table entry was outside the pool */
#define KVC_DEV_BAD_KEEP 8u     /* a keep position was outside its segment   */

/* Opaque CUDA stream handle (same object as cudaStream_t). */
typedef struct CUstream_st *kvc_stream_t;

/* The paged cache.  All pointers are device pointers. */
typedef struct kvc_cache {
    void *k_pool;         /* bf16 [L][num_pages][H][P][d]              */
    void *v_pool;         /* bf16 [L][num_pages][H][P][d]              */
    int32_t *tags;        /* int32 [L][num_pages][H][P]                */
    int32_t *block_table; /* int32 [batch][max_blocks]                 */
    int32_t *nblocks;     /* int32 [batch]: mapped blocks per sequence */
    int32_t num_layers;   /* L */
    int32_t num_pages;
    int32_t num_kv_heads; /* H */
    int32_t page_size;    /* P */
    int32_t head_dim;     /* d */
    int32_t max_blocks;
    int32_t batch;        /* B */
    float *aux;           /* fp32 [L][num_pages][H][P]: per-slot state that
                           * travels with its entry through kvc_compact (the
                           * LRFU values of kvc_lrfu_update, the bias beta
                           * of kvc_am_fit), or NULL */
} kvc_cache;

/* One segment per sequence, all host memory ([SE]: the application names the
 * range to prune).  seq_len[b] = slots in use by sequence b (its fill).  A
 * sequence with seg_start == seg_end takes no part in the call. */
typedef struct kvc_segments {
    const int32_t *seg_start; /* host [batch] */
    const int32_t *seg_end;   /* host [batch] */
    const int32_t *seq_len;   /* host [batch] */
    int32_t batch;
} kvc_segments;

/* Free-page stack of the page allocator (device memory).  Pop =
 * free_ids[--free_top], push = free_ids[free_top++]. */
typedef struct kvc_allocator {
    int32_t *free_ids; /* int32 [capacity] */
    int32_t *free_top; /* int32 [1]        */
    int32_t capacity;
} kvc_allocator;

/* Output of kvc_plan_compact, input of kvc_compact / kvc_free_pages.  The
 * caller allocates every buffer with the element counts of
 * kvc_plan_buffer_sizes.  A "physical slot" is page * P + offset.
 *   moves      int32 [L][H][Mtot][2]  (src, dst) physical slots; unit
 *              (l, h, b) owns entries [(l*H + h)*Mtot + moff_b, + m_b)
 *   move_count int32 [L][H][B]        valid moves of each unit
 *   dead       int32 [L][H][B][P]     holes left empty (tag becomes -1)
 *   dead_count int32 [L][H][B]
 *   freed      int32 [Ftot]           page ids to release, sequence order
 *   new_rows   int32 [B][max_blocks]  block-table rows after the release
 * Mtot = sum_b min(m_b, n_b); Ftot = sum_b (ceil(n_b/P) - ceil(m_b/P)). */
typedef struct kvc_plan {
    int32_t *moves;
    int32_t *move_count;
    int32_t *dead;
    int32_t *dead_count;
    int32_t *freed;
    int32_t *new_rows;
    int64_t moves_len; /* elements available in each buffer (checked) */
    int64_t units_len; /* move_count / dead_count length             */
    int64_t dead_len;
    int64_t freed_len;
    int64_t new_rows_len;
} kvc_plan;

typedef struct kvc_plan_sizes {
    int64_t moves_len;    /* int32 elements: 2 * L * H * Mtot */
    int64_t units_len;    /* L * H * B                         */
    int64_t dead_len;     /* L * H * B * P                     */
    int64_t freed_len;    /* Ftot                              */
    int64_t new_rows_len; /* B * max_blocks                    */
    int64_t Mtot;
    int64_t Ntot;
} kvc_plan_sizes;

/* ----------------------------------------------------------------- budget */

/* m = min(n, ceil(ratio * n)) -- keep ratio of [TE] (0.2 drops 80%), and
 * [SE]'s application-specified retain ratio.  The product is taken in
 * double with a 1e-9*n downward guard so that e.g. 0.07*100 gives 7.
 * Returns 0 for n <= 0 and clamps to [0, n]. */
int64_t kvc_budget_from_ratio(int64_t n, double ratio);

/* ActKV's ratchet budget after k growth steps ([ACT] budget paragraph):
 * min(30000, floor(512 * 1.75^k)).  k < 0 returns -1. */
int64_t kvc_budget_actkv(int32_t k);

/* ------------------------------------------------------------- hot path */

/* Bytes of workspace kvc_score needs for these segments and R proxy rows.
 * Returns KVC_OK and writes *bytes, or an argument error. */
kvc_status kvc_score_workspace_size(const kvc_cache *cache, const kvc_segments *segs, int32_t R,
                                    size_t *bytes);

/* Scores every key of every segment ([TE] score, [ACT] LSE recovery):
 *   L_ij  = scale * q_i . k_j  over the n keys of the segment
 *   LSE_i = log sum_j exp(L_ij)           (softmax over the segment)
 *   s_j   = sqrt((1/R) sum_i exp(2 (L_ij - LSE_i)))
 * q      bf16 [B][L][H][R][d], device: the R = q*g proxy rows of the g query
 *        heads that share KV head h (all rows of the group form Q).
 * scores out fp32 [L][H][Ntot]; sequence b at offset sum_{b'<b} n_b'.
 * lse    out fp32 [B][L][H][R] (natural log) or NULL.
 * ws     device workspace of kvc_score_workspace_size bytes.
 * Two tensor-core passes (bf16 operands, fp32 accumulation): the first
 * builds LSE from a running (offset, sum) per row, the second recomputes the logits and
 * accumulates alpha^2.  Keys are used as stored (no positional rotation).
 * scale must be finite and > 0. */
kvc_status kvc_score(const kvc_cache *cache, const kvc_segments *segs, const uint16_t *q,
                     int32_t R, float scale, float *scores, float *lse, void *ws, size_t ws_bytes,
                     kvc_stream_t stream);

/* The two passes of kvc_score as separate calls (same arguments, same
 * workspace; kvc_score == kvc_score_lse followed by kvc_score_alpha).
 *
 * kvc_score_lse: pass 1 only -- the per-row LSE over the segment ([ACT]:
 * log-sum-exp of the logits), kept in the workspace for kvc_score_alpha and
 * written to `lse` (fp32 [B][L][H][R], natural log) when it is not NULL.
 *
 * kvc_score_alpha: pass 2 only -- recomputes the logits and accumulates
 * alpha^2 into `scores`.  With lse == NULL it uses the LSE that the last
 * kvc_score_lse call left in `ws` (same cache, segments, R and scale).  With
 * a caller-supplied lse (fp32 [B][L][H][R], natural log) it normalises by
 * that instead -- e.g. the log-sum-exp a paged-attention kernel produced for
 * the same queries over the whole context ([ACT]: the LSE is a by-product of
 * paged attention), which skips pass 1 entirely. */
kvc_status kvc_score_lse(const kvc_cache *cache, const kvc_segments *segs, const uint16_t *q,
                         int32_t R, float scale, float *lse, void *ws, size_t ws_bytes,
                         kvc_stream_t stream);

kvc_status kvc_score_alpha(const kvc_cache *cache, const kvc_segments *segs, const uint16_t *q,
                           int32_t R, float scale, const float *lse, float *scores, void *ws,
                           size_t ws_bytes, kvc_stream_t stream);

/* kvc_score without a caller workspace.  (No counterpart on the pages: this is
 * an interface convenience.)  Some callers cannot allocate device memory for
 * the workspace: a serving engine whose allocator already owns the device's
 * memory for its page pool, code that must not enter the CUDA allocator on its
 * hot path, or a plugin that only receives the cache's pointers.  This entry
 * point takes the same inputs and outputs as kvc_score and puts the workspace
 * in a fixed 16 MiB device array inside the library; it calls no cudaMalloc,
 * cudaFree or allocating routine.
 *   - Every GPU that loads the library holds the 16 MiB array until the
 *     process exits.  A call whose workspace (kvc_score_workspace_size) is
 *     larger returns KVC_ERR_WORKSPACE and launches nothing.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and keeps it for the life of the process; make
 *     that first call before any stream capture.  A device reset while the
 *     library is loaded is not supported (see "Device reset" above).
 *   - All calls on a device share its array, which keeps the last call's
 *     contents (nothing in it needs to start at zero).  Calls whose kernels
 *     may overlap on the GPU (issued on different streams) race on the array:
 *     issue them on one stream. */
kvc_status kvc_score_noalloc(const kvc_cache *cache, const kvc_segments *segs, const uint16_t *q,
                             int32_t R, float scale, float *scores, float *lse, kvc_stream_t stream);

/* Bytes of workspace kvc_select_topm needs (may be 0). */
kvc_status kvc_select_workspace_size(const kvc_cache *cache, const kvc_segments *segs,
                                     const int32_t *m, size_t *bytes);

/* Keeps the top-m positions of every (layer, head, sequence) ([TE]):
 * m[b] (host, >= 0, clamped to n_b) positions with the highest score, equal
 * scores going to the lower position (decided on the fp32 scores), written
 * in ascending position order, segment-relative.
 * scores fp32 [L][H][Ntot] as written by kvc_score.
 * keep   out int32 [L][H][Mtot]; sequence b at offset sum_{b'<b} min(m_b', n_b').
 * Segments of at most 2^20 - 4096 = 1044480 positions (KVC_ERR_UNSUPPORTED
 * otherwise). */
kvc_status kvc_select_topm(const kvc_cache *cache, const kvc_segments *segs, const float *scores,
                           const int32_t *m, int32_t *keep, void *ws, size_t ws_bytes,
                           kvc_stream_t stream);

/* Element counts of the plan buffers for these segments and budgets. */
kvc_status kvc_plan_buffer_sizes(const kvc_cache *cache, const kvc_segments *segs,
                                 const int32_t *m, kvc_plan_sizes *out);

/* The conflict-free slot plan of [ACT], per (layer, head, sequence):
 * nb = ceil(n/P), X = ceil(m/P); the target region T is the last X blocks
 * of the segment; the k-th retained position before T (ascending) is paired
 * with the k-th hole of T (ascending slot; a hole is a slot of T holding no
 * retained entry, including slots past the segment end in its last block);
 * leftover holes are dead.  The first nb - X blocks are to be freed.
 * Reads the cache (block table) and keep; mutates nothing but the plan. */
kvc_status kvc_plan_compact(const kvc_cache *cache, const kvc_segments *segs, const int32_t *m,
                            const int32_t *keep, const kvc_plan *plan, kvc_stream_t stream);

/* Executes the plan as one parallel copy ([ACT]): K row, V row and tag of
 * every move; tag -1 on every dead hole.  Sources lie before T and
 * destinations inside it, so no entry is both.  Raw K/V bytes are copied
 * unmodified ([TE]).  Mutates k_pool, v_pool, tags. */
kvc_status kvc_compact(const kvc_cache *cache, const kvc_segments *segs, const int32_t *m,
                       const kvc_plan *plan, kvc_stream_t stream);

/* Returns the emptied blocks to the allocator ([ACT]): pushes plan->freed
 * (sequence order, ascending block order) onto the free stack, installs the
 * new block-table rows (later blocks shift down, vacated entries become -1)
 * and lowers nblocks[b] by ceil(n_b/P) - ceil(m_b/P).  Logical positions are
 * untouched: they travel in the tags ([SE] Chain Cache).  Must follow
 * kvc_plan_compact on the same stream; a stack overflow sets
 * KVC_DEV_FREE_STACK and pushes nothing. */
kvc_status kvc_free_pages(const kvc_cache *cache, const kvc_segments *segs, const int32_t *m,
                          const kvc_allocator *alloc, const kvc_plan *plan, kvc_stream_t stream);

/* ------------------------------------------------------------ ActKV scoring */

/* Action attention of every cached key ("ActKV 解剖", zhichai.net analysis of
 * ActKV, first component: the attention scores of all action tokens toward a
 * KV entry, gathered per entry):
 *   a_j = sum_i alpha_ij,  alpha_ij = exp(L_ij - LSE_i) over the segment,
 * with q holding the action tokens' query rows in the layout of kvc_score.
 * attn out fp32 [L][H][Ntot] (layout of kvc_score's scores); lse as in
 * kvc_score.  Same two tensor-core passes and workspace size as kvc_score. */
kvc_status kvc_score_action(const kvc_cache *cache, const kvc_segments *segs, const uint16_t *q,
                            int32_t R, float scale, float *attn, float *lse, void *ws,
                            size_t ws_bytes, kvc_stream_t stream);

/* One LRFU step of ActKV's eviction score (same page: entries within the top
 * 90% of action attention are action-critical; LRFU takes "hit by action
 * attention" as its reference signal, decay lambda = 0.5).  Per unit:
 * the action-critical entries are those with a_j >= tau, tau the largest
 * value whose entries a >= tau hold at least frac of the unit's total action
 * mass (the shortest prefix of the a-descending order reaching frac, boundary
 * ties included; nothing if the mass is 0 or frac = 0).  Then for every slot
 * of the segment: crf <- 2^-lambda * crf + hit in cache->aux (required), and
 * crf_out [L][H][Ntot] receives the new values (the eviction scores for
 * kvc_select_topm).  hits (uint8 [L][H][Ntot], may be NULL) receives the
 * flags.  Masses are summed in 2^-40 fixed point (64-bit integers), so the
 * result does not depend on the order of the sums.  frac in [0, 1], lambda
 * finite and >= 0; segments of at most 2^20 positions (KVC_ERR_UNSUPPORTED
 * beyond). */
kvc_status kvc_lrfu_update(const kvc_cache *cache, const kvc_segments *segs, const float *attn,
                           float frac, float lambda, float *crf_out, uint8_t *hits,
                           kvc_stream_t stream);

/* ------------------------------------------------- layout variants of eviction */

/* Layout-preserving eviction ("IntentKV: Cross-Turn Intent-Aware KV Cache
 * Pruning", section on layout-preserving eviction: an evicted position is
 * redirected to a sentinel dead slot with K = -10^4, V = 0, and surviving
 * rows keep their slots).  Every position of each segment that is not in
 * keep (the kvc_select_topm layout, ascending per unit) gets, in every
 * (layer, KV head): each of its d key elements = bf16(-10^4) (bit pattern
 * 0xC61C, value -9984), each value element = +0, tag = -1.  Retained
 * entries, slots past the segment end, the block table and the allocator
 * are untouched; no page is freed.  A keep entry outside [0, n) or out of
 * ascending order sets KVC_DEV_BAD_KEEP.  Mutates k_pool, v_pool, tags. */
kvc_status kvc_evict_sentinel(const kvc_cache *cache, const kvc_segments *segs, const int32_t *m,
                              const int32_t *keep, kvc_stream_t stream);

/* Buffer sizes of the fresh-page plan: those of kvc_plan_buffer_sizes except
 * freed_len = the sum of ceil(n_b/P) over sequences that keep fewer than all
 * of their n_b positions. */
kvc_status kvc_plan_fresh_buffer_sizes(const kvc_cache *cache, const kvc_segments *segs,
                                       const int32_t *m, kvc_plan_sizes *out);

/* Order-preserving compaction into fresh pages (an answer to the IntentKV
 * page's objection that in-place compaction renumbers positions): a sequence
 * keeping m_b < n_b positions takes X = ceil(m_b/P) pages from the free
 * stack, in pop order (pop k of the call hands out free_ids[free_top-1-k];
 * sequences ascending; every pop before any return), and in every unit its
 * r-th retained position moves to slot r of those pages (page r / P, offset
 * r % P), so physical order equals logical order; slots m_b .. X*P-1 of the
 * last fresh page are dead (tag -1).  All nb old blocks of the segment are
 * to be returned.  Fills *plan (moves, dead slots, the returned pages, the
 * new rows) for kvc_compact and kvc_commit_fresh; reads the allocator and
 * mutates nothing else.  A stack with fewer pages than the call pops sets
 * KVC_DEV_FREE_STACK and plans no moves.  The allocator must not change
 * between this call and kvc_commit_fresh. */
kvc_status kvc_plan_fresh(const kvc_cache *cache, const kvc_segments *segs, const int32_t *m,
                          const int32_t *keep, const kvc_allocator *alloc, const kvc_plan *plan,
                          kvc_stream_t stream);

/* Bookkeeping of the fresh-page compaction, after kvc_compact on the same
 * stream: pops the call's fresh pages, pushes every old block of the active
 * segments (sequences ascending, blocks ascending), replaces each active
 * segment's nb block-table entries by its X fresh pages (later entries shift
 * down by nb - X, vacated entries become -1) and lowers nblocks[b] by
 * nb - X.  If the device status word holds KVC_DEV_FREE_STACK (from the plan
 * or from this step's own capacity check) it changes nothing. */
kvc_status kvc_commit_fresh(const kvc_cache *cache, const kvc_segments *segs, const int32_t *m,
                            const kvc_allocator *alloc, const kvc_plan *plan, kvc_stream_t stream);

/* ------------------------------------------------------ Attention Matching */

/* Bytes of workspace kvc_am_fit needs: per (layer, head, sequence with m > 0)
 * about 4 * ((R + M) * (M + 4) + R * (d + 1) + M * (5 * d + 1)) bytes, M the
 * largest m among the (up to 128) sequences launched together, since their
 * fits share one layout (E [R][M+1], G [M][M+1], Y [R][d], LSE [R],
 * B [M][d], w [M], X [M][d], and B's sums over three more ranges of the R
 * rows [3][M][d]; rows padded to 4 floats, units to 256 bytes);
 * plus the workspace of the LSE pass (kvc_score_workspace_size) and
 * 4 * B * L * H * R bytes of row LSE; 0 when no sequence keeps an entry. */
kvc_status kvc_am_workspace_size(const kvc_cache *cache, const kvc_segments *segs, const int32_t *m,
                                 int32_t R, size_t *bytes);

/* Attention Matching on the survivors ([TE], section on the two compaction
 * families): with K_C the kept keys (`keep`, as written by kvc_select_topm),
 * fits an additive bias beta per kept key and compact values V_C so that the
 * compacted attention reproduces the full one on the proxy rows q:
 *   min_beta || exp(Q K_C^T + beta) 1_m - exp(Q K^T) 1_n ||^2
 *   min_V_C  || softmax(Q K_C^T + beta) V_C - softmax(Q K^T) V ||_F^2
 * (logits carry `scale`).  With w = exp(beta) >= 0 the first fit is
 * non-negative least squares; both run `sweeps` sweeps of cyclic coordinate
 * descent on their normal equations over the kept keys in ascending position
 * order, from token eviction's answer (beta = 0, V_C = the kept V rows), the
 * first projected onto w >= 0; the second uses the fitted beta.  sweeps in
 * [0, 1000]; 0 leaves token eviction's answer.  The full-attention targets
 * (LSE and softmax(Q K^T) V over all n keys) run on the tensor cores (bf16
 * Q, K and V as stored, fp32 accumulation, the probabilities in two bf16
 * parts); so do the Gram products of the normal equations, fp32-accurate
 * (each fp32 operand split into three bf16 parts, six partial products);
 * the coordinate descents run in fp32 on the CUDA cores.
 * Effects: every kept entry's V row becomes its V_C row (bf16, round to
 * nearest even) and, when cache->aux is not NULL, its per-slot state becomes
 * beta (-inf where w = 0: the key is masked); kvc_compact then moves both with
 * the entry.  K rows and tags are untouched.
 *   m     host [batch] budgets (clamped to n_b); every m_b <= 2048
 *   q     bf16 [B][L][H][R][d], R <= 4096, as for kvc_score
 *   lse   fp32 [B][L][H][R] natural-log LSE of the proxy rows over their
 *         segments, as kvc_score / kvc_score_lse write it for the same q, R and
 *         scale (the fit then runs no LSE pass of its own), or NULL: the fit
 *         runs the scoring LSE pass itself (same numbers)
 *   keep  int32 [L][H][Mtot] ascending segment positions (kvc_select_topm)
 *   beta  out fp32 [L][H][Mtot] or NULL
 *   vc    out fp32 [L][H][Mtot][d] (V_C before rounding) or NULL
 *   ws    kvc_am_workspace_size bytes, 256-byte aligned
 * A keep position outside its segment or out of ascending order sets
 * KVC_DEV_BAD_KEEP, a block-table entry outside the pool KVC_DEV_BAD_PAGE
 * (that entry is skipped). */
kvc_status kvc_am_fit(const kvc_cache *cache, const kvc_segments *segs, const int32_t *m,
                      const uint16_t *q, int32_t R, float scale, const float *lse, const int32_t *keep,
                      int32_t sweeps, float *beta, float *vc, void *ws, size_t ws_bytes,
                      kvc_stream_t stream);

/* -------------------------------------------------------------- helpers */

const char *kvc_status_string(kvc_status status);

/* Text of the last error returned on the calling thread ("" if none). */
const char *kvc_last_error(void);

/* Copies the device status word of the current device to *out (host) and,
 * if clear != 0, resets it.  Synchronises `stream`. */
kvc_status kvc_read_device_status(uint32_t *out, int32_t clear, kvc_stream_t stream);

/* Host-side consistency check of a cache's bookkeeping (host copies):
 * block-table entries of mapped blocks in [0, num_pages) and unique across
 * all sequences, unmapped entries -1, nblocks[b] <= max_blocks and
 * ceil(seq_len[b]/P) <= nblocks[b], free-stack entries in range, unique and
 * disjoint from mapped pages.  seq_len may be NULL.  Returns KVC_OK or
 * KVC_ERR_INVALID_ARG with the reason in kvc_last_error(). */
kvc_status kvc_validate_cache_host(const int32_t *block_table, const int32_t *nblocks,
                                   const int32_t *seq_len, int32_t batch, int32_t max_blocks,
                                   int32_t num_pages, int32_t page_size, const int32_t *free_ids,
                                   int32_t free_top);

/* Number of kernels the library has launched in this process (all devices)
 * since the last reset; reset != 0 returns the count and zeroes it. */
uint64_t kvc_launch_count(int32_t reset);

/* Library version string. */
const char *kvc_version(void);

/* Test support for failure detection; the pages have no counterpart.  Every
 * wait between the roles of a scoring kernel (producer, MMA issuer, epilogue)
 * is bounded: when one runs out the kernel records KVC_DEV_WAIT_TIMEOUT in
 * the device status word, waits (up to 2 s each) for the copies and MMAs it
 * has already issued, frees its tensor memory and returns, leaving the
 * context usable.  This call lets a test drive that path without faulting
 * anything: with stall_ns > 0, the scoring launches made afterwards
 * (kvc_score, kvc_score_lse, kvc_score_alpha, kvc_score_action,
 * kvc_score_noalloc) issue no proxy-row load and limit each wait between the
 * roles to stall_ns nanoseconds, so the MMA issuer's first wait can only run
 * out.  Such a call still returns KVC_OK (KVC_ERR_DEVICE_CHECK in checked
 * mode) and its outputs are undefined.  stall_ns = 0 restores normal
 * operation.  Process-wide, read when a call is made (a launch captured in a
 * CUDA graph keeps the value it was captured with).  Returns
 * KVC_ERR_INVALID_ARG unless 0 <= stall_ns <= 1e10. */
kvc_status kvc_debug_stall_scoring(int64_t stall_ns);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
