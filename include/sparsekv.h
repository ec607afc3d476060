/*
 * sparsekv.h -- C interface of the GB300 sparse paged-KV decode attention library.
 *
 * One decode step of attention over a paged KV cache, with query-aware page selection:
 *
 *   kv_build_page_stats    per-page, per-KV-head element-wise min/max of the keys
 *   kv_score_pages         an upper bound of q.k over each page, summed over a GQA group
 *   kv_select_topk         top-k pages per (sequence, KV head) under a keep ratio/budget
 *   kv_sparse_decode_attn  split-K softmax attention over the selected pages -> partials
 *   kv_merge_splits        log-sum-exp merge of the (m, l, acc) partials -> output, lse
 *   kv_dropped_mass        diagnostic: dense attention mass of the pages not selected
 *   kv_decode_step         the four per-step calls above in one call, on a workspace
 *
 * Sources, by page title and section:
 *   [ENTMAX]  "EntmaxKV: Support-Aware Decoding for Entmax Attention", abstract: pages are
 *             scored against the query from cheap per-page statistics before any page is
 *             read; the output error is governed by the dropped mass delta.
 *   [SPARDA]  "SparDA: Sparse Decoupled Attention for Efficient Long-Context LLM
 *             Inference", section 3.1 (per-head relevance summed inside a GQA group into
 *             one shared score), appendix A (the top-k operator over block scores),
 *             appendix C (a fixed block budget).
 *   [BYTEX]   "Where Activation Sparsity and KV-Cache Sparsity Cross in LLM Decoding",
 *             abstract and Table 11 (dense and sparse decoding read the cache through the
 *             same split-K attention kernel; dense is that kernel with every page kept),
 *             Tables 16-17 (keep ratios r_KV).
 *   [PRHS]    "Near-Oracle KV Selection via Pre-hoc Sparsity for Long-Context Inference",
 *             abstract (top-k KV selection; delta = attention mass of discarded entries).
 *
 * Conventions for every call
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless the comment
 *     says "host". The library allocates no device memory and keeps no per-call state:
 *     the caller provides every output and workspace buffer.
 *   - Every call is asynchronous on the given stream (0 = the legacy default stream).
 *   - Host-detectable argument errors return KV_ERR_INVALID_ARG, KV_ERR_UNSUPPORTED or
 *     KV_ERR_MISALIGNED and launch nothing. A failed launch returns KV_ERR_CUDA.
 *   - Device-detected faults in the DATA (a page-table entry outside [0, num_phys_pages),
 *     a sequence longer than its page-table row, a selected index outside the sequence,
 *     a keep count above k_max, an asynchronous copy that did not land in time) never
 *     trap: the kernel skips the bad access, records a flag in a per-device error word
 *     and finishes. kv_check_device_errors() reports and clears that word.
 *   - Supported shapes: head_dim 64 or 128; page_size 16, 32 or 64; group size
 *     G = num_q_heads / num_kv_heads in {1, 2, 4, 8}; dtype bf16 or fp32. Anything else
 *     returns KV_ERR_UNSUPPORTED.
 *
 * Layouts (row-major, innermost last)
 *   k_pool, v_pool  [num_phys_pages][num_kv_heads][page_size][head_dim]   dtype
 *   page_table      [batch][page_table_stride] int32; entry p of row b is the physical
 *                   page of logical page p of sequence b; only p < ceil(len_b/page_size)
 *                   are read.
 *   seq_lens        [batch] int32 tokens, the current decode token included.
 *   q               [batch][num_q_heads][head_dim] dtype; query head h reads KV head
 *                   h / G (consecutive query heads share a KV head).
 *   stats           [num_phys_pages][num_kv_heads][2][head_dim] dtype; [..][0][:] = min,
 *                   [..][1][:] = max over the page's valid tokens.
 *   scores          [batch][num_kv_heads][scores_stride] float32.
 *   sel_idx         [batch][num_kv_heads][sel_stride] int32 logical page indices,
 *                   ascending; sel_cnt [batch][num_kv_heads] int32 entries used.
 *   part_acc        [batch][num_q_heads][num_splits][head_dim] float32
 *   part_ml         [batch][num_q_heads][num_splits][2] float32 = (m, l)
 *   out             [batch][num_q_heads][head_dim] float32; lse [batch][num_q_heads].
 *
 * Alignment: k_pool, v_pool, stats and q must be 16-byte aligned (pages are moved with
 * bulk asynchronous copies); otherwise KV_ERR_MISALIGNED.
 */
#ifndef SPARSEKV_H_
#define SPARSEKV_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kv_status {
  KV_OK = 0,
  KV_ERR_INVALID_ARG = -1,   /* a null pointer, a non-positive size, inconsistent sizes */
  KV_ERR_UNSUPPORTED = -2,   /* a shape or dtype outside the supported set */
  KV_ERR_CUDA = -3,          /* a CUDA runtime call or launch failed */
  KV_ERR_WORKSPACE = -4,     /* workspace null or smaller than the *_workspace_size */
  KV_ERR_BAD_INDEX = -5,     /* device-detected: bad page, length, index or keep count */
  KV_ERR_TIMEOUT = -6,       /* device-detected: a bounded wait ran out */
  KV_ERR_MISALIGNED = -7     /* a buffer is not 16-byte aligned */
} kv_status;

typedef enum kv_dtype { KV_BF16 = 0, KV_FP32 = 1 } kv_dtype;

/* num_splits value of kv_decode_step that asks for the one-launch step. */
#define KV_SPLITS_ONE_LAUNCH (-1)

/* Device-side error flags (bit mask) behind kv_check_device_errors(). */
enum {
  KV_DEVERR_BAD_PAGE = 1,    /* page-table entry outside [0, num_phys_pages) */
  KV_DEVERR_BAD_LEN = 2,     /* seq_len < 0 or above page_table_stride * page_size */
  KV_DEVERR_BAD_SEL = 4,     /* selected index outside [0, n_pages) or sel_cnt > stride */
  KV_DEVERR_KEEP = 8,        /* keep count above k_max (clamped to k_max) */
  KV_DEVERR_TIMEOUT = 16     /* bounded wait on an asynchronous copy ran out */
};

/* The paged cache. All pointers are device pointers owned by the caller. */
typedef struct kv_cache_desc {
  const void* k_pool;           /* [num_phys_pages][num_kv_heads][page_size][head_dim] */
  const void* v_pool;           /* same layout as k_pool */
  int32_t dtype;                /* kv_dtype of k_pool, v_pool, q and stats */
  int32_t num_phys_pages;
  int32_t num_kv_heads;
  int32_t page_size;            /* tokens per page: 16, 32 or 64 */
  int32_t head_dim;             /* 64 or 128 */
  int32_t batch;                /* sequences */
  const int32_t* page_table;    /* [batch][page_table_stride] */
  int32_t page_table_stride;    /* >= max over b of ceil(seq_lens[b] / page_size) */
  const int32_t* seq_lens;      /* [batch] tokens, current token included */
} kv_cache_desc;

/* Human-readable name of a kv_status value (static string, never NULL). */
const char* kv_status_string(int32_t status);

/* Library interface version (major * 100 + minor). */
int32_t kv_version(void);

/*
 * kv_build_page_stats -- [ENTMAX] per-page statistics.
 * For every mapped page (b, p < ceil(len_b/PS)) and KV head g, writes the element-wise
 * min and max of the keys of the page's valid tokens (min(PS, len_b - p*PS) of them) to
 * stats[page_table[b][p]][g][0|1][:]. Values are copied exactly (no rounding). Rows of
 * unmapped physical pages are not written. Reads every mapped key once; run it after a
 * prefill, not per step.
 * stats: device, [num_phys_pages][num_kv_heads][2][head_dim] of the cache dtype.
 * phys_pages: NULL to build every mapped page; otherwise device int32[n_phys], STRICTLY
 * ASCENDING physical page indices, and only the mapped pages whose physical index is in the
 * list are (re)built (e.g. the pages a chunked prefill just wrote); every other row of
 * stats is left as it was, and listed pages that no sequence maps are not written. Cost:
 * one page-table read per mapped page plus the keys of the listed ones. A list entry outside
 * [0, num_phys_pages) or out of order is flagged (KV_DEVERR_BAD_PAGE; which pages are then
 * rebuilt is unspecified). n_phys outside [0, num_phys_pages] returns KV_ERR_INVALID_ARG;
 * n_phys = 0 with a list does nothing.
 */
kv_status kv_build_page_stats(const kv_cache_desc* cache, void* stats,
                              const int32_t* phys_pages, int32_t n_phys, cudaStream_t stream);

/*
 * kv_build_page_stats_fp8 -- the statistics of kv_build_page_stats stored in one byte each
 * (the compressed page statistics motivated by [BYTEX]'s selector key cache quantised to few
 * bits), with outward rounding so that the score stays an upper bound ([ENTMAX]).
 * For each mapped (page P, KV head g) row of 2*head_dim values (min row, max row):
 *   e = smallest integer >= -126 with max |x| <= 448 * 2^e over the row (0 if all zero),
 *   stats_exp[P][g] = e,
 *   min byte = E4M3 byte of the largest value v with v * 2^e <= min,
 *   max byte = E4M3 byte of the smallest value v with v * 2^e >= max,
 * E4M3 being the OCP "FN" byte (bias 7, 3 mantissa bits, subnormals, largest 448, no
 * infinity; zero is written as 0x00). Decoded min <= true min and decoded max >= true max.
 * stats_fp8: device, [num_phys_pages][num_kv_heads][2][head_dim] bytes, 16-byte aligned;
 * stats_exp: device, [num_phys_pages][num_kv_heads] int8. Unmapped pages are not written.
 */
kv_status kv_build_page_stats_fp8(const kv_cache_desc* cache, void* stats_fp8,
                                  int8_t* stats_exp, cudaStream_t stream);

/*
 * kv_append_token -- [ENTMAX] the cache grows by one token per decode step; this call adds
 * that token and keeps the page statistics current without re-reading the cache.
 * For every sequence b with seq_lens[b] > 0 (seq_lens already counts the new token), the
 * token goes to position t = seq_lens[b] - 1: slot t % page_size of logical page
 * t / page_size, which page_table must already map. Its key and value rows
 * k_new[b][g][:], v_new[b][g][:] are written to k_pool and v_pool (the descriptor's pool
 * pointers are written through), and the page's statistics become the element-wise min/max
 * of the old ones and the key (a page's first token, slot 0, resets them to the key). The
 * result equals kv_build_page_stats of the grown cache bit for bit.
 * k_new, v_new: device [batch][num_kv_heads][head_dim] of the cache dtype.
 * stats: device [num_phys_pages][num_kv_heads][2][head_dim] of the cache dtype.
 */
kv_status kv_append_token(const kv_cache_desc* cache, const void* k_new, const void* v_new,
                          void* stats, cudaStream_t stream);

/*
 * kv_score_pages -- [ENTMAX] query-aware page score, [SPARDA] summed over a GQA group.
 * scores[b][g][p] = sum over query heads h of group g, over d, of
 *                   max(q[b][h][d] * mn[d], q[b][h][d] * mx[d])
 * with (mn, mx) = stats of physical page page_table[b][p], KV head g. Each term bounds
 * q_d * k_d for every key of the page, so the per-head sum bounds q.k over the page. The
 * softmax scale is left out (it does not change the order). Computed in float32.
 * Entries p >= ceil(len_b / PS) are not written. scores_stride >= page_table_stride.
 */
kv_status kv_score_pages(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                         const void* stats, float* scores, int32_t scores_stride,
                         cudaStream_t stream);

/*
 * kv_score_pages_fp8 -- kv_score_pages from the statistics of kv_build_page_stats_fp8: the
 * same formula with mn, mx the decoded values byte * 2^e (an upper bound of the exact-stats
 * score, as the decoded box contains the exact one). Computed in float32.
 */
kv_status kv_score_pages_fp8(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                             const void* stats_fp8, const int8_t* stats_exp, float* scores,
                             int32_t scores_stride, cudaStream_t stream);

/*
 * kv_select_topk -- [PRHS], [SPARDA] appendix A: top-k pages of each (b, g) group.
 * n_b = ceil(seq_lens[b] / page_size). The keep count k_b is
 *   keep[b]                                   if keep is not NULL (device [batch]),
 *   min(n_b, budget_pages)                    else if budget_pages > 0,
 *   n_b                                       else if keep_ratio >= 1,
 *   min(n_b, max(1, ceil(keep_ratio*n_b - 1e-9)))   otherwise (ratio in (0, 1)),
 * and 0 when n_b = 0 (the ratio rule is evaluated in double precision, so that e.g.
 * 0.2 * 5 keeps 1 page, not 2). k_b above k_max is clamped to k_max and flagged
 * (KV_DEVERR_KEEP); a negative keep[b] is taken as 0.
 * Pages are ranked by (score descending, page index ascending) -- ties go to the lower
 * page index -- and the k_b best are written to sel_idx[b][g][0..k_b) in ASCENDING page
 * order, with sel_cnt[b][g] = k_b. Scores must not be NaN.
 * scores: device [batch][num_kv_heads][scores_stride] float32 (as kv_score_pages writes).
 * sel_idx: device [batch][num_kv_heads][k_max]; sel_cnt: device [batch][num_kv_heads].
 */
kv_status kv_select_topk(const float* scores, int32_t scores_stride, const int32_t* seq_lens,
                         int32_t page_size, int32_t batch, int32_t num_kv_heads,
                         const int32_t* keep, double keep_ratio, int32_t budget_pages,
                         int32_t k_max, int32_t* sel_idx, int32_t* sel_cnt,
                         cudaStream_t stream);

/*
 * kv_select_structured -- kv_select_topk with forced pages: [SPARDA] section 3.1 and
 * appendix A join initial blocks, a local window of the most recent blocks and top-k blocks.
 * For each group the first sink_pages and the last local_pages pages (the set F, clipped to
 * the group's n pages) are always kept, the keep count becomes max(k_b, |F|) (then clamped
 * to k_max as in kv_select_topk), and the remaining places go to the best-scoring pages
 * outside F under kv_select_topk's order. scores may be NULL: every page outside F then ties,
 * so the lowest-indexed ones fill the remaining places; with sink_pages = 0 and
 * local_pages = k this is the KV-window baseline of [BYTEX] Tables 3 and 11 (keep the last k
 * pages, no scoring). Arguments are otherwise those of kv_select_topk; at least one of a
 * keep rule and a forced page count must be given.
 */
kv_status kv_select_structured(const float* scores, int32_t scores_stride,
                               const int32_t* seq_lens, int32_t page_size, int32_t batch,
                               int32_t num_kv_heads, const int32_t* keep, double keep_ratio,
                               int32_t budget_pages, int32_t sink_pages, int32_t local_pages,
                               int32_t k_max, int32_t* sel_idx, int32_t* sel_cnt,
                               cudaStream_t stream);

/*
 * kv_sparse_decode_attn -- [BYTEX] split-K decode attention over selected pages.
 * For each (b, g) the selected list (sel_idx[b][g][0..sel_cnt[b][g]), or every page
 * 0..n_b-1 when sel_idx is NULL: the dense baseline through the same kernel) is cut into
 * num_splits consecutive runs of whole 64-token tiles: with p = 64 / page_size pages a tile
 * and T = ceil(cnt / p) tiles, split s takes list positions
 * [min(cnt, floor(s*T/num_splits)*p), min(cnt, floor((s+1)*T/num_splits)*p)), so the runs
 * differ by at most one tile and only the list's last tile is partial. For each query head h
 * of the group and split s, over the
 * valid tokens t of the run's pages (tokens at or past len_b are masked):
 *   x_t = sm_scale * q[b][h] . k_t,  m = max x_t,  l = sum exp(x_t - m),
 *   acc = sum exp(x_t - m) v_t
 * written as part_ml[b][h][s] = (m, l), part_acc[b][h][s][:] = acc. An empty split
 * writes (m, l) = (-inf, 0) and acc = 0. Accumulation is float32.
 * num_splits >= 1 (kv_auto_num_splits gives a value that fills the GPU).
 * sel_stride: row stride of sel_idx (the k_max used by kv_select_topk); ignored when
 * sel_idx is NULL. sel_cnt may be NULL only when sel_idx is NULL.
 */
kv_status kv_sparse_decode_attn(const kv_cache_desc* cache, const void* q,
                                int32_t num_q_heads, float sm_scale, const int32_t* sel_idx,
                                const int32_t* sel_cnt, int32_t sel_stride,
                                int32_t num_splits, float* part_acc, float* part_ml,
                                cudaStream_t stream);

/*
 * kv_score_select -- kv_score_pages followed by kv_select_topk (keep = NULL) in ONE launch.
 * Writes scores (as kv_score_pages), sel_idx [batch][num_kv_heads][k_max] and sel_cnt
 * [batch][num_kv_heads] (as kv_select_topk: same keep rule, same order, same ascending
 * output). The block of each group that finishes its scores last runs the group's
 * selection. counters: device [batch][num_kv_heads] int32, zero before the first call;
 * every call returns them to zero. keep_ratio > 0 or budget_pages > 0. The group's keys
 * must fit one block's shared memory: page_table_stride up to about 50,000 pages on GB300
 * (KV_ERR_UNSUPPORTED beyond; kv_score_pages + kv_select_topk have no such limit).
 */
kv_status kv_score_select(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                          const void* stats, double keep_ratio, int32_t budget_pages,
                          int32_t k_max, float* scores, int32_t scores_stride,
                          int32_t* counters, int32_t* sel_idx, int32_t* sel_cnt,
                          cudaStream_t stream);

/*
 * kv_decode_attn_merge -- kv_sparse_decode_attn followed by kv_merge_splits in ONE launch,
 * for bf16 caches. Arguments and per-split results are those of kv_sparse_decode_attn
 * (sel_idx NULL = every page, the dense baseline); the last of a group's split CTAs to
 * finish merges the group's partials into out/lse by the formula of kv_merge_splits.
 * counters: device [batch][num_kv_heads] int32, zero before the first call; every call
 * returns them to zero. part_acc must be 16-byte and part_ml 8-byte aligned
 * (KV_ERR_MISALIGNED). num_splits is bounded by the merge's on-chip buffer
 * (KV_ERR_UNSUPPORTED above it; over 700 splits for every supported shape).
 */
kv_status kv_decode_attn_merge(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                               float sm_scale, const int32_t* sel_idx, const int32_t* sel_cnt,
                               int32_t sel_stride, int32_t num_splits, float* part_acc,
                               float* part_ml, int32_t* counters, float* out, float* lse,
                               cudaStream_t stream);

/*
 * kv_select_decode_attn -- kv_select_topk, kv_sparse_decode_attn and kv_merge_splits in ONE
 * kernel, for bf16 caches. Each of a group's num_splits CTAs selects its own run of the
 * kept pages from the group's score row (the rule and order of kv_select_topk with keep =
 * NULL; the run split of kv_sparse_decode_attn), attends over it, writes its partial to
 * part_acc/part_ml, and the group's last CTA merges the partials into out/lse (the formula
 * of kv_merge_splits). With scores = NULL every page is kept: the dense baseline through
 * the same kernel. counters: device [batch][num_kv_heads] int32, zero before the first call;
 * every call returns them to zero. counters = NULL: no merge -- the call only writes the
 * partials (for kv_merge_splits to merge) and out/lse are not touched (they may be NULL). sel_idx [batch][num_kv_heads][k_max] and sel_cnt
 * [batch][num_kv_heads] receive the selection when not NULL (sparse calls only). The group's
 * pages must fit the in-kernel selection (page_table_stride at most 21440 pages for
 * head_dim 128, 9152 for 64) and the splits its merge; otherwise KV_ERR_UNSUPPORTED.
 * part_acc must be 16-byte and part_ml 8-byte aligned (KV_ERR_MISALIGNED).
 */
kv_status kv_select_decode_attn(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                                float sm_scale, const float* scores, int32_t scores_stride,
                                double keep_ratio, int32_t budget_pages, int32_t k_max,
                                int32_t num_splits, float* part_acc, float* part_ml,
                                int32_t* counters, float* out, float* lse, int32_t* sel_idx,
                                int32_t* sel_cnt, cudaStream_t stream);

/*
 * kv_merge_splits -- log-sum-exp merge of the split partials ([BYTEX] split-K).
 * M = max_s m_s; L = sum_s l_s exp(m_s - M); out = sum_s acc_s exp(m_s - M) / L;
 * lse = M + log L (natural log). Splits with m = -inf carry no mass; if every split is
 * empty, out = 0 and lse = -inf. lse may be NULL.
 */
kv_status kv_merge_splits(const float* part_acc, const float* part_ml, int32_t batch,
                          int32_t num_q_heads, int32_t num_splits, int32_t head_dim,
                          float* out, float* lse, cudaStream_t stream);

/*
 * kv_auto_num_splits -- host: a split count for a cache of this shape when each (b, g) group
 * keeps about pages_per_group pages: the most splits whose CTAs (batch * num_kv_heads * S)
 * all fit the device's resident CTA slots at once (no partial second wave), at least one,
 * at most one per two 64-token tiles, and at least what the merge's split limit needs.
 * Returns >= 1, or a negative kv_status on a bad argument.
 */
int32_t kv_auto_num_splits(const kv_cache_desc* cache, int32_t num_q_heads,
                           int32_t pages_per_group);

/*
 * kv_dropped_mass -- [PRHS], [ENTMAX] diagnostic probe, not part of a decode step.
 * delta[b][h] = sum over valid tokens of pages NOT in sel_idx[b][g] of exp(x_t - M)
 *               / sum over all valid tokens of exp(x_t - M),  x_t = sm_scale * q.k_t,
 * M the max over all valid tokens; 0 for an empty sequence. Reads every key of every
 * mapped page. workspace: device, at least kv_dropped_mass_workspace_size() bytes.
 */
kv_status kv_dropped_mass(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                          float sm_scale, const int32_t* sel_idx, const int32_t* sel_cnt,
                          int32_t sel_stride, float* delta, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream);

size_t kv_dropped_mass_workspace_size(const kv_cache_desc* cache, int32_t num_q_heads);

/*
 * kv_decode_step -- one sparse decode step: kv_score_pages, kv_select_topk,
 * kv_sparse_decode_attn and kv_merge_splits on a caller workspace. With keep_ratio >= 1
 * and budget_pages <= 0 it is the dense step (every page, no scoring or selection).
 * k_max bounds the keep count (and sizes the workspace).
 * num_splits > 0: the four calls run with that many splits; 0: the four calls with
 * kv_auto_num_splits' count; KV_SPLITS_ONE_LAUNCH: for bf16 caches whose (sequence, KV head)
 * groups fit one wave of thread-block clusters, the whole step is ONE launch -- a cluster per
 * group scores, selects, attends and merges in on-chip memory (distributed shared memory
 * between the cluster's CTAs), each CTA being one split (other shapes fall back to the four
 * calls). Both paths give the same selection (bit for bit) and outputs equal up to float32
 * rounding of the merge.
 * out: device [batch][num_q_heads][head_dim] float32; lse: [batch][num_q_heads] or NULL.
 * For bf16 caches: groups of up to 16384 pages (page_table_stride, and within
 * kv_select_decode_attn's limit) run kv_score_pages, then an attention kernel whose CTAs each
 * select their own run; longer ones kv_score_select, then the attention over the list; the
 * dense step is the attention kernel alone. With fewer than 8 splits the attention kernel's
 * last CTA per group merges (two launches, one for the dense step); with 8 or more the merge
 * is a kernel of its own, chained to the attention kernel by programmatic dependent launch
 * (kv_decode_step_plan tells which).
 * workspace: device, at least kv_decode_step_workspace_size() bytes, 256-byte aligned, ZERO-
 * FILLED ONCE before its first use: it starts with two int32 counters per group, at offsets
 * that depend only on batch * num_kv_heads, which the kernels return to zero after every
 * step, so one workspace serves sparse and dense calls and any k_max or split count (as
 * long as it is large enough). After a sparse call it holds the step's selection:
 * sel_idx [batch][num_kv_heads][k_max] int32 at byte offset
 * A = 2 * round256(batch * num_kv_heads * 4) + round256(batch * num_kv_heads *
 * round4(page_table_stride) * 4), and sel_cnt [batch][num_kv_heads] int32 at
 * A + round256(batch * num_kv_heads * k_max * 4), where round256(x) and round4(x) round x
 * up to a multiple of 256 and of 4 (the layout kv_dropped_mass can be fed from).
 */
kv_status kv_decode_step(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                         float sm_scale, const void* stats, double keep_ratio,
                         int32_t budget_pages, int32_t k_max, int32_t num_splits,
                         float* out, float* lse, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);

size_t kv_decode_step_workspace_size(const kv_cache_desc* cache, int32_t num_q_heads,
                                     int32_t k_max, int32_t num_splits);

/*
 * kv_decode_step_graph_create / _launch / _destroy -- kv_decode_step captured once into a CUDA
 * graph, for a serving loop that runs the same step every token: each launch then costs the
 * host one graph launch instead of the argument checks, planning and kernel launches of
 * kv_decode_step. create makes one uncaptured kv_decode_step call (checking the arguments
 * and doing every first-use set-up; the workspace must therefore be zero-filled as for
 * kv_decode_step), then captures the same call on a private stream and instantiates it.
 * Every pointer and size is baked into the graph: the caller keeps all the buffers (cache
 * descriptor's pools, page table, lengths, q, stats, out, lse, workspace) alive and in place
 * while the graph exists, and changes only their CONTENTS between launches (the new query,
 * appended tokens and grown lengths, within the page table's capacity). The step's plan and
 * split count are those of the capture. launch runs the step on `stream` (asynchronous, like
 * kv_decode_step); launches of one graph must not overlap on the GPU (they share the
 * workspace). destroy frees the graph (NULL is accepted). create returns kv_decode_step's
 * status for bad arguments, KV_ERR_CUDA if capture or instantiation fails; *graph is NULL
 * then. The graph holds host and driver resources only; no device buffer is allocated.
 * q_host (host, page-locked, batch * num_q_heads * head_dim elements of the cache dtype)
 * and out_host (host, page-locked, batch * num_q_heads * head_dim float32) may be NULL;
 * when given, one launch per token carries the query in and the output back. A buffer the
 * device addresses in place (page-locked memory under unified addressing, as
 * cudaPointerGetAttributes reports) is read (q_host) or written (out_host) by the step's
 * kernels themselves over the host link, and q (or out) is then not used; any other is
 * copied: q_host into q before the step, out into out_host after it.
 */
typedef struct kv_step_graph kv_step_graph;
kv_status kv_decode_step_graph_create(const kv_cache_desc* cache, const void* q,
                                      int32_t num_q_heads, float sm_scale, const void* stats,
                                      double keep_ratio, int32_t budget_pages, int32_t k_max,
                                      int32_t num_splits, float* out, float* lse,
                                      void* workspace, size_t workspace_bytes,
                                      const void* q_host, float* out_host,
                                      kv_step_graph** graph);
kv_status kv_decode_step_graph_launch(kv_step_graph* graph, cudaStream_t stream);
kv_status kv_decode_step_graph_destroy(kv_step_graph* graph);

/*
 * kv_decode_step_fp8 -- kv_decode_step scoring from FP8 statistics (kv_build_page_stats_fp8)
 * instead of statistics in the cache's dtype: the same plans, workspace and outputs, with
 * kv_score_pages_fp8's scores. KV_SPLITS_ONE_LAUNCH runs the automatic plan instead (the
 * one-launch kernel reads cache-dtype statistics). Dense calls ignore the statistics.
 */
kv_status kv_decode_step_fp8(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                             float sm_scale, const void* stats_fp8, const int8_t* stats_exp,
                             double keep_ratio, int32_t budget_pages, int32_t k_max,
                             int32_t num_splits, float* out, float* lse, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/*
 * kv_decode_step_plan -- host, launches nothing: the kernels kv_decode_step runs for these
 * arguments (a KV_PLAN_* value, or a negative kv_status), and in *splits (if not NULL) its
 * split count (the cluster size for KV_PLAN_ONE_LAUNCH). All plans give the same selection
 * and outputs equal up to float32 rounding of the merge.
 */
typedef enum {
  KV_PLAN_FOUR_KERNELS = 0,            /* kv_score_pages, kv_select_topk,
                                          kv_sparse_decode_attn, kv_merge_splits */
  KV_PLAN_SCORE_THEN_SELECT_ATTN = 1,  /* kv_score_pages, kv_select_decode_attn */
  KV_PLAN_SCORE_SELECT_THEN_ATTN = 2,  /* kv_score_select, kv_decode_attn_merge */
  KV_PLAN_DENSE_ATTN_MERGE = 3,        /* kv_decode_attn_merge with every page */
  KV_PLAN_DENSE_TWO_KERNELS = 4,       /* kv_sparse_decode_attn, kv_merge_splits */
  KV_PLAN_ONE_LAUNCH = 5,              /* one thread-block cluster per group */
  KV_PLAN_SCORE_THEN_SELECT_ATTN_THEN_MERGE = 6,  /* kv_score_pages, the attention kernel
                                          selecting per CTA (partials only), kv_merge_splits */
  KV_PLAN_SCORE_SELECT_THEN_ATTN_THEN_MERGE = 7   /* kv_score_select, kv_sparse_decode_attn
                                          over the list, kv_merge_splits */
} kv_plan;
int32_t kv_decode_step_plan(const kv_cache_desc* cache, int32_t num_q_heads, double keep_ratio,
                            int32_t budget_pages, int32_t k_max, int32_t num_splits,
                            int32_t* splits);

/*
 * kv_decode_step_static -- kv_decode_step without a workspace argument, for callers that
 * cannot allocate device memory on the decode path (a plain C or plugin host with no
 * device allocator of its own, or a serving loop that must not call cudaMalloc per token,
 * since that can synchronise the device or fail under memory pressure mid-step). The pages
 * have no counterpart of this call: it only moves the scratch of kv_decode_step into the
 * library. It runs kv_score_pages, kv_select_topk, kv_sparse_decode_attn and kv_merge_splits
 * (no per-group counters, so nothing in the array has to keep a value between calls): the
 * selection is kv_decode_step's bit for bit and the outputs equal up to float32 rounding of
 * the merge. num_splits <= 0 (KV_SPLITS_ONE_LAUNCH included) means kv_auto_num_splits' count.
 * Scratch: one file-scope __device__ array of KV_STATIC_SCRATCH_BYTES that every GPU loading
 * the library holds until exit. CUDA loads the module holding it lazily, so the first call on
 * a device loads that module, reserves the array (which can fail under memory pressure,
 * returning KV_ERR_CUDA, or synchronise) and looks up its device address
 * (cudaGetSymbolAddress, that device current): make that first call at start-up, before any
 * stream capture. All calls share the array and it keeps the last call's contents: calls
 * that overlap on the GPU race and must be serialised by the caller. Nothing in it needs to
 * start at zero. Limit: this call's own scratch -- batch * num_kv_heads * page_table_stride
 * float32 scores, batch * num_kv_heads * k_max int32 indices (1 for a dense call),
 * batch * num_kv_heads int32 counts, and batch * num_q_heads * S * (head_dim + 2) float32
 * split partials, each rounded up to a multiple of 256 bytes -- above
 * KV_STATIC_SCRATCH_BYTES returns KV_ERR_WORKSPACE and launches nothing. Once its array is
 * in place, a call allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine).
 */
#define KV_STATIC_SCRATCH_BYTES (8u << 20)
kv_status kv_decode_step_static(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                                float sm_scale, const void* stats, double keep_ratio,
                                int32_t budget_pages, int32_t k_max, int32_t num_splits,
                                float* out, float* lse, cudaStream_t stream);

/*
 * Entmax decoding over selected pages -- the next-step row after [ENTMAX] (abstract):
 * alpha-entmax gives exact zeros, so attention over the selected pages equals full attention
 * once the selection holds the support, and a Gaussian-aware selector estimates the entmax
 * threshold from the page statistics so that the kept budget adapts to the scores.
 * Readings: alpha = 1.5; with z_t = sm_scale * q . k_t / 2 the weights are
 * p_t = max(z_t - tau, 0)^2 with sum p_t = 1 over the attended tokens (tau in z units).
 *
 * kv_entmax_page_moments -- per query head h and logical page p (stats as kv_build_page_stats):
 *   zb = (sm_scale/2) sum_d max(q_d mn_d, q_d mx_d)            (upper bound of z over the page)
 *   cz = (sm_scale/2) q . (mn + mx)/2                          (box-centre z)
 *   vz = (sm_scale/2)^2 sum_d q_d^2 (mx_d - mn_d)^2 / 12      (within-box variance of z)
 * written to [batch][num_q_heads][stride] float32 each (entries past a sequence untouched).
 */
kv_status kv_entmax_page_moments(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                                 const void* stats, float sm_scale, float* zb, float* cz,
                                 float* vz, int32_t stride, cudaStream_t stream);

/*
 * kv_entmax_select -- Gaussian-aware threshold selection per (b, g) group: for each query
 * head, with n_p the valid tokens of page p and N = sum n_p,
 *   mu = sum n_p cz_p / N,  sigma^2 = sum n_p (cz_p - mu)^2 / N + sum n_p vz_p / N,
 *   tau_hat solving N * E[max(Z - tau_hat, 0)^2] = 1 for Z ~ N(mu, sigma^2)
 * (closed form s^2((u^2+1) Phi(u) + u phi(u)), u = (mu - tau)/s, solved in float by Newton
 * on its logarithm). A page is kept if zb > tau_hat for some head of the group, and each head's
 * highest-zb page (the lower index on ties) is always kept. Kept pages go to
 * sel_idx[b][g][...] ascending, their count to sel_cnt[b][g]; more than k_max is flagged
 * (KV_DEVERR_KEEP) and the first k_max are kept. tau_hat [batch][num_q_heads] may be NULL.
 */
kv_status kv_entmax_select(const float* zb, const float* cz, const float* vz, int32_t stride,
                           const int32_t* seq_lens, int32_t page_size, int32_t batch,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t k_max,
                           int32_t* sel_idx, int32_t* sel_cnt, float* tau_hat,
                           cudaStream_t stream);

/*
 * kv_entmax_decode_attn -- 1.5-entmax attention of each decode query over the valid tokens of
 * its group's selected pages (sel_idx NULL: every page, the dense entmax baseline):
 * out[b][h] = sum_t max(z_t - tau, 0)^2 v_t with tau solved exactly over those tokens
 * (tau[b][h] written if tau is not NULL; NaN and a zero output for a group with no token).
 * K is read for the attended pages, V only for tokens with a nonzero weight.
 * workspace: device, kv_entmax_attn_workspace_size() bytes (the candidate lists: 8 bytes
 * per attended token slot and query head, plus 8 bytes per split), 16-byte aligned.
 * KV_ERR_UNSUPPORTED when the pools hold more than 2^32 - 1 rows (num_phys_pages *
 * num_kv_heads * page_size): the candidate lists keep a token's row in 32 bits.
 */
size_t kv_entmax_attn_workspace_size(const kv_cache_desc* cache, int32_t num_q_heads,
                                     int32_t sel_stride);
kv_status kv_entmax_decode_attn(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                                float sm_scale, const int32_t* sel_idx, const int32_t* sel_cnt,
                                int32_t sel_stride, float* out, float* tau, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/*
 * kv_entmax_decode_step -- kv_entmax_page_moments, kv_entmax_select and kv_entmax_decode_attn
 * on a caller workspace (256-byte aligned, kv_entmax_decode_step_workspace_size() bytes).
 * After the call the workspace holds the selection: with M = round256(batch * num_q_heads *
 * page_table_stride * 4), sel_idx [batch][num_kv_heads][k_max] int32 at byte 3M and sel_cnt
 * [batch][num_kv_heads] at 3M + round256(batch * num_kv_heads * k_max * 4).
 */
size_t kv_entmax_decode_step_workspace_size(const kv_cache_desc* cache, int32_t num_q_heads,
                                            int32_t k_max);
kv_status kv_entmax_decode_step(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                                float sm_scale, const void* stats, int32_t k_max, float* out,
                                float* tau, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream);

/*
 * kv_workspace_size -- host, launches nothing: the bytes of device workspace that call `op`
 * needs for these arguments -- the same value as that call's own *_workspace_size function,
 * which it dispatches to (KV_OP_DECODE_STEP: kv_decode_step_workspace_size(cache,
 * num_q_heads, k_max, num_splits), also for kv_decode_step_fp8; KV_OP_DROPPED_MASS:
 * kv_dropped_mass_workspace_size(cache, num_q_heads); KV_OP_ENTMAX_DECODE_ATTN:
 * kv_entmax_attn_workspace_size(cache, num_q_heads, k_max as sel_stride, 0 = every page);
 * KV_OP_ENTMAX_DECODE_STEP: kv_entmax_decode_step_workspace_size(cache, num_q_heads,
 * k_max)). Arguments a given op does not use are ignored. Every other call of this library
 * takes no workspace. Returns 0 for an unknown op or a bad argument.
 */
typedef enum {
  KV_OP_DECODE_STEP = 0,
  KV_OP_DROPPED_MASS = 1,
  KV_OP_ENTMAX_DECODE_ATTN = 2,
  KV_OP_ENTMAX_DECODE_STEP = 3
} kv_op;
size_t kv_workspace_size(int32_t op, const kv_cache_desc* cache, int32_t num_q_heads,
                         int32_t k_max, int32_t num_splits);

/*
 * kv_check_device_errors -- synchronises `stream`, reads and clears the current device's
 * error word. Returns KV_OK, KV_ERR_TIMEOUT (a bounded wait ran out) or KV_ERR_BAD_INDEX
 * (any other flag). If flags is not NULL (host), the raw KV_DEVERR_* mask is stored.
 */
kv_status kv_check_device_errors(cudaStream_t stream, int32_t* flags);

/*
 * kv_set_wait_limit_ns -- host: limit, in nanoseconds of the GPU's global timer, of every
 * device-side wait on an asynchronous copy (default 2e9). After it runs out the kernel
 * flags KV_DEVERR_TIMEOUT, drains its own copies (again bounded) and returns.
 */
kv_status kv_set_wait_limit_ns(uint64_t limit_ns);

/*
 * kv_selftest_wait_timeout -- launches one block that waits, with the production bounded
 * wait, on a barrier that nothing ever completes, using `limit_ns` as the limit. Used to
 * test the timeout path: a following kv_check_device_errors() must return KV_ERR_TIMEOUT.
 */
kv_status kv_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPARSEKV_H_ */
