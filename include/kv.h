/*
 * kv.h -- C ABI of the B300 (sm_103a) paged KV-cache library: one decode step
 * of grouped-query attention over a block-table KV cache, and the page
 * budgeting step (query summaries, page scoring, top-k retention,
 * compress-or-grow, compaction, append).
 *
 * Sources for what each call computes:
 *  [PKV] aissential.tech, "PersistentKV: Page-Aware Decode Scheduling for
 *        Long-Context LLM Serving on Commodity GPUs" -- Summary, Method:
 *        native block-table decode attention for GQA that reuses each K/V
 *        tile across the grouped query heads and runs a compact workqueue of
 *        non-empty (sequence, KV-head, split) tasks.
 *  [GP]  mlsanity.com, "GrowPage: On-Demand KV Budgeting for Efficient LLM
 *        Reasoning Serving" -- Abstract; aitrending.vip GrowPage summary --
 *        Technical Details: query summaries at a short and a long time
 *        scale, their attention working sets compared to track demand,
 *        compress-or-grow at every capacity boundary, on top of
 *        PagedAttention's page abstraction.
 *  [EKV] paperlayer.ai, "Elastic KV Cache for LLM Serving" -- section 2:
 *        fixed-size KV blocks handed out from an integer free list.
 *
 * Conventions shared by every call
 *  - Pointers marked (device) are device memory owned by the caller; (host)
 *    pointers are host memory (pinned for asynchronous copies).  The library
 *    never allocates memory and never keeps a pointer past the call.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *    enqueue work and return; none synchronises except kv_get_status.
 *  - Return value: KV_OK, or a negative KV_E* code for an argument rejected
 *    on the host (nothing was enqueued).  Errors found on the device (a bad
 *    page id, an exhausted free list, ...) are recorded in the status word of
 *    the workspace `ws` and read back with kv_get_status; the kernels never
 *    trap and never read or write outside the buffers described here.
 *  - 16-bit element types: dtype KV_F16 (IEEE binary16) or KV_BF16.
 *    Floating outputs are fp32.
 *  - Layouts (row-major):
 *      q            [B][Hq][d]                    16-bit
 *      k_pool/v_pool [num_pages][Hkv][page_size][d] 16-bit (page-major, then
 *                   KV head: one (page, head) tile is page_size*d contiguous
 *                   elements, all heads of a page are contiguous)
 *      block_table  [B][max_pages] int32: logical page j of sequence b lives
 *                   in pool page block_table[b][j]; entries at j >= ceil(L_b /
 *                   page_size) are never read (-1 padding is customary)
 *      seq_lens     [B] int32, tokens held by each sequence (L_b >= 0)
 *    Query head hq attends with KV head hq / (Hq / Hkv) (contiguous groups).
 *  - Supported shapes: page_size 16; d in {64, 128}.  The fused decode kernel
 *    takes Hq / Hkv in {1, 2, 4, 8} and Hkv <= 8, the tensor-core engine any
 *    Hq / Hkv <= 64 (and any Hkv).  Others return KV_EINVAL.
 *  - Workspace: `ws` is caller-allocated device memory of at least the size
 *    the matching *_workspace_size function returns, 256-byte aligned.  Its
 *    first 256 bytes hold the status word.  One workspace may serve several
 *    calls that run in order on one stream (kv_decode excepted: see
 *    kv_decode_workspace_size); calls that overlap on the device must not
 *    share one.  Zero it once before first use (kv_workspace_reset).
 */
#ifndef PAGED_KV_B300_KV_H
#define PAGED_KV_B300_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KV_OK 0
#define KV_EINVAL (-1)     /* bad argument (host) or bad length (device) */
#define KV_EBADPAGE (-2)   /* a page id in use is < 0 or >= num_pages */
#define KV_ENOSPACE (-3)   /* free list holds fewer pages than needed */
#define KV_EWORKSPACE (-4) /* workspace too small for the work found */
#define KV_ECUDA (-5)      /* a CUDA runtime call failed */
#define KV_EFULL (-6)      /* a block-table row has no room for a new page */
#define KV_ETIMEOUT (-7)   /* a kernel's bounded wait gave up (never expected) */

#define KV_F16 0
#define KV_BF16 1

/* pages_per_split value that selects the tensor-core decode engine (see
 * kv_decode). */
#define KV_DECODE_TENSOR_CORE (-1)

/* Text for a status code (static storage). */
const char *kv_status_string(int code);

/* The CUDA runtime call behind the most recent KV_ECUDA returned on the
 * calling host thread, with the runtime's error name and text; "" if none.
 * Thread-local storage owned by the library, valid until the next call that
 * fails on this thread. */
const char *kv_last_error(void);

/* Bytes of the workspace header (the status word); the minimum workspace. */
size_t kv_status_workspace_size(void);

/* Zero the first ws_bytes bytes of a workspace (at least the status word)
 * on `stream`.  A new workspace must be zeroed once before its first call;
 * after a KV_ETIMEOUT zero it again before reusing it. */
int kv_workspace_reset(void *ws, size_t ws_bytes, void *stream);

/* Synchronise `stream`, return the first device-side error recorded in `ws`
 * since the last call (KV_OK if none) and clear it. */
int kv_get_status(void *ws, void *stream);

/* ------------------------------------------------------------------------ */
/* Decode [PKV].                                                              */
/* ------------------------------------------------------------------------ */

/* Number of decode workers (resident CTAs, one per split-chunk at a time) on
 * the current device for this shape; the automatic split size spreads the
 * batch's pages evenly over them. */
int kv_decode_num_workers(int Hq, int Hkv, int d, int page_size, int dtype);

/* Workspace bytes kv_decode needs for a batch of B sequences whose tables are
 * max_pages wide.  pages_per_split as passed to kv_decode (0 = automatic;
 * KV_DECODE_TENSOR_CORE: the tensor-core engine, whose size also covers the
 * fused kernel with the automatic split, and whose scratch lies past the
 * fused kernel's merge tickets for every split size).
 * Besides scratch, a decode workspace keeps one merge ticket per (sequence,
 * KV head) that must read zero when a call starts: every kv_decode that
 * completes leaves them zero, so a decode workspace stays valid across
 * calls as long as no other call writes into it (give kv_decode a workspace
 * of its own; the budgeting calls use theirs as scratch).  A counter found
 * non-zero is reported as KV_EWORKSPACE. */
size_t kv_decode_workspace_size(int B, int Hq, int Hkv, int d, int max_pages, int page_size,
                                int pages_per_split);

/* One decode step.  For every sequence b and query head hq (h = hq / G):
 *   s_t   = scale * <q[b][hq], k_t>      over tokens t < L_b of the paged cache
 *   lse   = ln sum_t exp(s_t)            (natural log, scale included)
 *   out   = sum_t exp(s_t - lse) v_t
 * out [B][Hq][d] fp32 (device), lse [B][Hq] fp32 (device).  L_b = 0 gives
 * out = 0 and lse = -inf.
 * Work split: the non-empty pages of the batch, laid end to end, are cut into
 * chunks of `pages_per_split` pages (0 = automatic: ceil(W / workers), at
 * least 8, W = total pages); each (sequence, chunk) overlap is one split, and
 * each split is one task per KV head (the queue kv_build_workqueue
 * materialises).  A task streams each (page, KV head) tile once from HBM and
 * reuses it for all G = Hq/Hkv query heads; splits of one sequence are
 * recombined by a log-sum-exp merge done by whichever split finishes last.
 * One kernel launch (two for B > 1024: a page-offset pass first).
 * pages_per_split = KV_DECODE_TENSOR_CORE selects the tensor-core engine
 * instead (d = 64 or 128, page_size 16, G <= 64; else KV_EINVAL): the same split
 * rule with the automatic chunk, one CTA per chunk streaming whole pages by
 * TMA tensor copies, Q K^T and P V on mma.sync (fp32 accumulation), and a
 * merge kernel for the split sequences (kv_attend_multi with T = 1).  Both
 * engines compute the same function; which is faster depends on the
 * workload (kv_decode_tune).
 * Device errors: KV_EBADPAGE (an entry in [0, ceil(L_b/16)) outside
 * [0, num_pages); page 0 is read in its place), KV_EINVAL (L_b < 0 or more
 * pages than max_pages), KV_EWORKSPACE, KV_ETIMEOUT. */
int kv_decode(const void *q, const void *k_pool, const void *v_pool, int num_pages,
              const int32_t *block_table, int max_pages, const int32_t *seq_lens, int B,
              int page_size, int Hq, int Hkv, int d, int dtype, float scale,
              int pages_per_split, float *out, float *lse, void *ws, size_t ws_bytes,
              void *stream);

/* Several new query tokens per sequence (a prefill chunk, or the drafted
 * tokens of a speculative step) over the same pool and block table: the T
 * queries of sequence b are its last T cached tokens (their K/V already
 * appended), and query i attends causally to tokens [0, L_b - T + 1 + i):
 *   s_t = scale * <q[b][i][hq], k_t>,  lse = ln sum_t exp(s_t),
 *   out[b][i][hq] = sum_t exp(s_t - lse) v_t;
 * a query with no token to attend to gets out = 0 and lse = -inf.
 * q [B][T][Hq][d] 16-bit, out [B][T][Hq][d] fp32, lse [B][T][Hq] fp32
 * (device).  Other arguments and errors as kv_decode; the workspace is
 * kv_attend_multi_workspace_size bytes (give it its own).  The tensor-core
 * engine (d = 64 or 128, page_size 16, G <= 64; else KV_EINVAL) serves up to
 * 64 / G tokens per pass over the pages (T * G <= 64: one pass for all T
 * tokens; T = 1 is kv_decode's KV_DECODE_TENSOR_CORE engine); larger T runs
 * as ceil(T * G / 64) consecutive passes over chunks of at most 64 / G
 * tokens, so each page is streamed that many times.  The chunks use as few
 * 16-row blocks as the T tokens need, spread evenly over the passes (where G
 * divides 16; otherwise every pass but the last is full). */
size_t kv_attend_multi_workspace_size(int B, int T, int Hq, int Hkv, int d, int max_pages,
                                      int page_size, int pages_per_split);
int kv_attend_multi(const void *q, const void *k_pool, const void *v_pool, int num_pages,
                    const int32_t *block_table, int max_pages, const int32_t *seq_lens, int B,
                    int T, int page_size, int Hq, int Hkv, int d, int dtype, float scale,
                    int pages_per_split, float *out, float *lse, void *ws, size_t ws_bytes,
                    void *stream);

/* Calibration among this library's own decode variants (the adaptive policy
 * of [PKV] Summary picks an engine per workload by measurement; here the
 * variants are the fused kernel's split sizes and the tensor-core engine):
 * runs kv_decode on the given inputs once per candidate pages_per_split
 * (0 = automatic, KV_DECODE_TENSOR_CORE = tensor-core engine) untimed, then `reps` (<= 64)
 * times timed with CUDA events on `stream`, writes the microseconds per
 * candidate (mean of the middle half of its sorted times) to
 * us[n_candidates] (host) and the fastest candidate to
 * *best (host).  Synchronises `stream`; out/lse hold the last call's result.
 * `ws` must be sized for every candidate (kv_decode_workspace_size with the
 * smallest positive candidate covers all positive ones, and the size for
 * KV_DECODE_TENSOR_CORE covers it and the automatic one: pass the larger).
 * `flush` (device, flush_bytes; NULL for none): a buffer more than twice the
 * size of the L2 cache, overwritten and then read back over its first half
 * before every timed call (outside the events), so the candidates are timed
 * with their inputs in HBM and with no dirty lines of the flush left in L2 to
 * write back, as a step that follows ordinary work finds them; without it
 * they are timed back to back, warm in L2.  The buffer's contents are
 * scratch. */
int kv_decode_tune(const void *q, const void *k_pool, const void *v_pool, int num_pages,
                   const int32_t *block_table, int max_pages, const int32_t *seq_lens, int B,
                   int page_size, int Hq, int Hkv, int d, int dtype, float scale,
                   const int32_t *candidates, int n_candidates, int reps, float *out, float *lse,
                   float *us, int32_t *best, void *ws, size_t ws_bytes, void *flush,
                   size_t flush_bytes, void *stream);

/* Profiling aid: the next kv_decode (or kv_decode_hostio) issued from the
 * calling host thread records `event_before` (a cudaEvent_t) on its stream
 * just before the attention kernel and `event_after` just after it, so the
 * kernel's own duration can be timed with CUDA events.  One-shot; NULL
 * events disarm it. */
int kv_profile_next_decode(void *event_before, void *event_after);

/* Testing aid for the failure path (no counterpart on the pages): while `ns`
 * is non-zero, every decode launched afterwards from this process (kv_decode
 * with either engine, kv_attend_multi, kv_decode_hostio, kv_decode_noalloc)
 * makes each consumer warp first wait `ns` nanoseconds on a barrier that
 * nothing completes.  The wait runs out, and the kernel takes the way out
 * every bounded wait takes: KV_ETIMEOUT in the status word, the producer
 * stops issuing copies and waits for those in flight, and the outputs of
 * non-empty sequences are left unwritten.  No GPU fault is involved.  0 (the
 * default) turns it off.  A workspace used
 * in this mode may hold partial merge state: reset it (kv_workspace_reset)
 * before the next call. */
int kv_test_consumer_timeout(unsigned long long ns);

/* Workspace bytes for kv_decode_hostio: kv_decode's plus staging for q, the
 * block table, seq_lens, out and lse. */
size_t kv_decode_hostio_workspace_size(int B, int Hq, int Hkv, int d, int max_pages,
                                       int page_size, int pages_per_split);

/* kv_decode with the per-step inputs and outputs in host memory: copies
 * h_q, h_block_table, h_seq_lens (host) into the workspace, runs kv_decode
 * against the device-resident pools, and delivers out/lse into h_out and
 * h_lse (host), all enqueued on `stream`.  Page-locked host buffers (which
 * the device can address) are used in place: one copy kernel reads the three
 * inputs, and the decode kernels write out/lse straight into h_out/h_lse
 * (h_out 16-byte aligned; otherwise they are staged and copied back).
 * Pageable buffers take one cudaMemcpyAsync each.  The host buffers must
 * stay valid, and h_out/h_lse unread, until the stream reaches the end of
 * the call. */
int kv_decode_hostio(const void *h_q, const void *k_pool, const void *v_pool, int num_pages,
                     const int32_t *h_block_table, int max_pages, const int32_t *h_seq_lens,
                     int B, int page_size, int Hq, int Hkv, int d, int dtype, float scale,
                     int pages_per_split, float *h_out, float *h_lse, void *ws, size_t ws_bytes,
                     void *stream);

/* kv_decode for callers that cannot allocate device memory.  The paper has
 * no counterpart: this is a library convenience.  Some callers only ever
 * hold their own input and output buffers -- a host framework that plans and
 * owns every device allocation, or a plugin interface that forbids
 * allocating on the hot path (cudaMalloc synchronises the device) -- and so
 * cannot hand kv_decode a workspace.  This entry point takes the same inputs
 * and outputs as kv_decode, plus `status`, one int32 in device memory that
 * the call sets to 0 and then to the first device-side error (the codes
 * kv_get_status would return); it allocates nothing and calls no cudaMalloc,
 * cudaFree or allocating library routine.
 * Its scratch is one 16 MiB array in the library's device memory, present on
 * every device that loads the library until the process exits.  The first
 * call on a device looks up the array's device address (once per device and
 * CUDA context: after a cudaDeviceReset the next call looks it up again);
 * make that first call before any stream capture.  A batch whose scratch
 * (the size kv_decode_workspace_size reports) exceeds 16 MiB is rejected
 * with KV_EWORKSPACE and nothing is enqueued; with the automatic split this
 * holds every supported shape up to tens of thousands of sequences.  Every
 * call zeroes the part of the array it relies on (its merge tickets
 * included), so a call that stopped early -- KV_ETIMEOUT -- leaves nothing
 * that disturbs the next one, and unlike kv_decode this entry point never
 * reports KV_EWORKSPACE for leftover tickets.  All calls share the array:
 * calls whose work overlaps on the GPU (other streams, other host threads)
 * race and must be serialised by the caller.  B = 0 enqueues only the
 * zeroing of *status. */
int kv_decode_noalloc(const void *q, const void *k_pool, const void *v_pool, int num_pages,
                      const int32_t *block_table, int max_pages, const int32_t *seq_lens, int B,
                      int page_size, int Hq, int Hkv, int d, int dtype, float scale,
                      int pages_per_split, float *out, float *lse, int32_t *status, void *stream);

/* The decode workqueue on its own (for inspection and tests).  With
 * chunk = pages_per_split (> 0) or the automatic size for n_workers workers
 * (pages_per_split = 0): writes, in (b, split, h) order, one 8 x int32 record
 * per task: b, h, split, nsplit_b, page_begin, page_end (pages of b), chunk
 * index, L_b.  chunk_begin [nchunks + 1]: first (b, split) group of each
 * chunk.  seq_group_begin [B], seq_nsplit [B].  meta [5] int32: tasks,
 * groups, chunk, nchunks, W.  Capacities max_tasks / max_chunks (entries);
 * overflow -> KV_EWORKSPACE in the status word.  All arrays (device); `ws`
 * of kv_workqueue_workspace_size(B) bytes holds the status word and scratch. */
size_t kv_workqueue_workspace_size(int B);
int kv_build_workqueue(const int32_t *seq_lens, int B, int Hkv, int page_size, int max_pages,
                       int pages_per_split, int n_workers, int32_t *tasks, int max_tasks,
                       int32_t *chunk_begin, int max_chunks, int32_t *seq_group_begin,
                       int32_t *seq_nsplit, int32_t *meta, void *ws, void *stream);

/* ------------------------------------------------------------------------ */
/* Page budgeting [GP].  Build's instantiation of the summaries the pages     */
/* describe without a formula (every value that decides an integer is fp32    */
/* with the operation order stated, so results are reproducible bit for bit):*/
/*   query summaries: per KV head the group-mean query g (sum over the G      */
/*     query heads in ascending order, then / G), and two EMAs               */
/*     ema = (a * ema) + ((1 - a) * g), a = a_fast or a_slow;                */
/*   page key summaries: per (page, KV head, channel) mean (sum of the 16    */
/*     slots in order, / 16), min and max;                                    */
/*   page score S_u(j) = sum_h sum_c [u*mean + max(u*min, u*max)], summed    */
/*     per lane l (channels l*d/32 .. +d/32, heads then channels ascending)  */
/*     and across lanes by xor-butterfly 16, 8, 4, 2, 1.                      */
/* ------------------------------------------------------------------------ */

/* ema [B][2][Hkv][d] fp32 (device), index 0 fast, 1 slow; first != 0
 * initialises both to g.  q [B][Hq][d] (device). */
int kv_update_query_summaries(const void *q, int B, int Hq, int Hkv, int d, int dtype,
                              float a_fast, float a_slow, int first, float *ema, void *stream);

/* active [B] uint8 (device).  mode 0: ceil(L_b/16) > budget[b] (sequences
 * over budget); mode 1: capacity boundary, L_b > 0, L_b % 16 == 0 and
 * L_b / 16 >= budget[b]. */
int kv_mark_active(const int32_t *seq_lens, const int32_t *budget, int B, int page_size, int mode,
                   uint8_t *active, void *stream);

/* summ [num_pages][Hkv][3][d] fp32 (device): for each listed pool page,
 * mean/min/max over its 16 slots.  page_ids [n] (device). */
int kv_page_summaries(const void *k_pool, int num_pages, const int32_t *page_ids, int n, int Hkv,
                      int page_size, int d, int dtype, float *summ, void *ws, size_t ws_bytes,
                      void *stream);

/* Same summaries for the last page of every active sequence
 * (block_table[b][L_b/16 - 1]), i.e. the page that has just filled. */
int kv_summarize_last_pages(const void *k_pool, int num_pages, const int32_t *block_table,
                            int max_pages, const int32_t *seq_lens, const uint8_t *active, int B,
                            int Hkv, int page_size, int d, int dtype, float *summ, void *ws,
                            size_t ws_bytes, void *stream);

/* scores [B][max_pages][2] fp32 (device): S_fast, S_slow of each resident
 * logical page of each active sequence (active NULL = all); -inf for
 * j >= ceil(L_b/16); inactive rows untouched. */
int kv_score_pages(const float *query_summaries, const float *page_key_summaries, int num_pages,
                   const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                   const uint8_t *active, int B, int Hkv, int d, int page_size, float *scores,
                   void *ws, size_t ws_bytes, void *stream);

#define KV_SELECT_TOPK 0
#define KV_SELECT_BOUNDARY 1

size_t kv_select_workspace_size(int B, int max_pages);

/* Top-k retention and compress-or-grow.  n = ceil(L_b/16); forced pages
 * F = {j < n_first} U {j >= n - n_last}; candidates C = the rest; ranking by
 * larger key first, equal keys by lower logical index; R = S_fast + S_slow.
 * KV_SELECT_TOPK: keep = F U top_(budget[b]-|F|)(C, R) for active rows.
 * KV_SELECT_BOUNDARY: w = ceil(ws_frac*|C|) (fp32, clipped to [1, |C|]);
 *   drift D = |top_w(C, S_fast) \ top_w(C, S_slow)|; a row wants to grow iff
 *   D > delta*w (fp32) or C is empty; grows are granted in ascending b while
 *   fewer than *free_top (device) have been granted: grow[b] = 1,
 *   budget[b] += 1, keep every page.  Otherwise keep = F U top_(n-1-|F|)(C, R).
 * Inactive rows keep every page.  keep_mask [B][max_pages] uint8, grow [B]
 * uint8, drift [B] int32 (may be NULL), budget [B] int32 in/out (device). */
int kv_select_pages(const float *scores, const int32_t *seq_lens, const uint8_t *active,
                    int32_t *budget, int B, int max_pages, int page_size, int n_first, int n_last,
                    float delta, float ws_frac, int mode, const int32_t *free_top,
                    uint8_t *keep_mask, uint8_t *grow, int32_t *drift, void *ws, size_t ws_bytes,
                    void *stream);

/* num_pages: the pool's page count when kv_compact will be given refcnt
 * (shared pages), else 0. */
size_t kv_compact_workspace_size(int B, int max_pages, int num_pages, int token_granular);

/* Stable compaction [GP] with the free list of [EKV]: the kept tokens of
 * each sequence (keep_mask [B][max_pages] per page, or [B][max_pages*16]
 * per token when token_granular) fill new slots 0, 1, ... in order.  New
 * page m reuses old page j when it holds exactly j's first tokens at the
 * same slots (page masks always do: no K/V moves); otherwise it takes a
 * fresh page popped from free_list[*free_top - 1 - i] in (b, m) order and
 * the tokens' K and V (all heads) are copied there.  Old pages not reused
 * are then pushed in (b, j) order.  block_table rows are rewritten (-1
 * padded), seq_lens become the kept counts, *free_top is updated.
 * free_list has num_pages entries (device).
 * Shared pages (prefix caching, which GrowPage keeps [GP]): refcnt [num_pages]
 * int32 (device, or NULL when every page belongs to one sequence) holds each
 * pool page's number of block-table references.  A fresh page gets 1; every
 * old page not reused loses one reference, in (b, j) order, and is pushed
 * when none is left (by the reference that takes it to zero).  Kept pages are
 * never written, so a page other sequences still use is left as it is.
 * Device errors: KV_ENOSPACE (nothing is changed), KV_EBADPAGE. */
int kv_compact(int32_t *block_table, int max_pages, int32_t *seq_lens, const uint8_t *keep_mask,
               int token_granular, void *k_pool, void *v_pool, int num_pages, int32_t *free_list,
               int32_t *free_top, int32_t *refcnt, int B, int Hkv, int d, int page_size, int dtype,
               void *ws, size_t ws_bytes, void *stream);

size_t kv_append_workspace_size(int B);

/* Append one token per sequence: K/V (k_new, v_new [B][Hkv][d], device) go
 * to slot L_b % 16 of page block_table[b][L_b / 16]; when L_b % 16 == 0 that
 * page is first popped from the free list (pops in ascending b).  Then
 * L_b += 1.  With refcnt (shared pages, as for kv_compact; NULL = none), a
 * sequence whose partly filled last page is shared copies it first
 * (copy-on-write): in ascending b, while the page has more than one
 * reference left, the sequence pops a fresh page (same pop order), the
 * page's filled slots (K and V, all heads) are copied there, its table entry
 * moves to the fresh page and the shared page loses one reference; the last
 * sharer writes in place.  Popped pages get count 1.  All copies are made
 * before any token is written.  Device errors (nothing is changed):
 * KV_ENOSPACE, KV_EFULL, KV_EBADPAGE. */
int kv_append(const void *k_new, const void *v_new, void *k_pool, void *v_pool, int num_pages,
              int32_t *block_table, int max_pages, int32_t *seq_lens, int32_t *free_list,
              int32_t *free_top, int32_t *refcnt, int B, int Hkv, int d, int page_size, int dtype,
              void *ws, size_t ws_bytes, void *stream);

/* The budgeting part of one steady-state step [GP] in two launches (the step
 * and a copy of the token's K/V rows), for a batch without shared pages: the
 * same results, bit for bit, as the calls
 *   kv_update_query_summaries (first = 0; skipped when update_ema = 0),
 *   kv_mark_active (mode 1), kv_summarize_last_pages, kv_score_pages,
 *   kv_select_pages (KV_SELECT_BOUNDARY), kv_compact (page masks),
 *   kv_append
 * issued in that order on a valid state (every table entry in use is a pool
 * page, lengths within the rows, finite scores).  Sixteen work items per
 * sequence at a capacity boundary (one for any other), taken in turn by a
 * resident grid, form its updated EMAs and share its page scores (the item
 * owning the last page summarises it first); the last of them to finish
 * writes the EMAs, ranks the candidates under both summaries (working sets,
 * drift) and compacts the row unless it wants to grow; the last sequence to
 * finish grants the grows in ascending b, compacts the rows that got no
 * page, pushes the freed pages in (b, j) order and plans the append, whose
 * K/V rows (k_new, v_new [B][Hkv][d]) a second kernel copies.  No block
 * waits on another.  Arguments as in those calls;
 * d in {64, 128}; `ws` of kv_budget_step_workspace_size bytes, zeroed before
 * its first use and used by no other call: it keeps per-sequence counters
 * that each call leaves at zero (reset it after a call that failed).  Device
 * errors as those calls report them. */
size_t kv_budget_step_workspace_size(int B, int max_pages);
int kv_budget_step(const void *q, const void *k_new, const void *v_new, void *k_pool,
                   void *v_pool, int num_pages, int32_t *block_table, int max_pages,
                   int32_t *seq_lens, int32_t *budget, int B, int Hq, int Hkv, int d,
                   int page_size, int dtype, float a_fast, float a_slow, int update_ema,
                   int n_first, int n_last, float delta, float ws_frac, float *ema, float *summ,
                   float *scores, uint8_t *active, uint8_t *keep_mask, uint8_t *grow,
                   int32_t *drift, int32_t *free_list, int32_t *free_top, void *ws,
                   size_t ws_bytes, void *stream);

/* Hand pool pages [first_page, first_page + n) to the free list (the
 * integer free list of [EKV] section 2): pushed highest id first, so the
 * following pops (kv_append, kv_compact) take them in ascending order.  This
 * is how the pages of an elastic pool's growth (kv_vmm_pool_resize) become
 * available to a budgeted sequence that grows.  free_list has `capacity`
 * entries and *free_top (device) is its height; if the pages do not fit,
 * KV_ENOSPACE goes to the status word of `ws` (kv_status_workspace_size
 * bytes) and nothing changes. */
int kv_free_list_push(int first_page, int n, int32_t *free_list, int capacity, int32_t *free_top,
                      void *ws, void *stream);

/* ------------------------------------------------------------------------ */
/* Elastic page pool [EKV, section 3]: one reserved virtual address range     */
/* per pool whose physical backing grows and shrinks at its top, so pages     */
/* never move, block tables stay valid and the kernels are unchanged.  This   */
/* is the one part of the library that allocates device memory, on request.   */
/* ------------------------------------------------------------------------ */

/* Reserve max_bytes (rounded up to the allocation granularity) of virtual
 * address space on `device`; nothing is backed yet.  *pool: opaque handle;
 * *base: the range's device address (page p of a pool of page_bytes pages
 * lives at base + p * page_bytes); *granularity (may be NULL): the size unit
 * of every resize.  Errors: KV_EINVAL, KV_ECUDA (kv_last_error names the
 * driver call). */
int kv_vmm_pool_create(int device, size_t max_bytes, void **pool, void **base,
                       size_t *granularity);

/* Back the first `bytes` (rounded up to the granularity) of the range.
 * Growing maps one new physical allocation directly above the mapped part;
 * shrinking unmaps and frees whole earlier growths from the top, so the
 * result may stay above `bytes` (*mapped, may be NULL, reports it).  The
 * contents of pages that stay mapped are untouched.  Synchronous with respect
 * to the device (the driver calls are); the caller must not shrink under
 * pages that are still referenced or in use by running kernels. */
int kv_vmm_pool_resize(void *pool, size_t bytes, size_t *mapped);

/* Bytes currently backed (0 for a NULL pool). */
size_t kv_vmm_pool_mapped(void *pool);

/* Unmap and free everything and release the address range. */
int kv_vmm_pool_destroy(void *pool);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_B300_KV_H */
