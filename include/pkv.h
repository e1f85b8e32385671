/*
 * pkv.h -- C ABI of libpkv: paged-KV grouped-query decode attention on GB300.
 *
 * Method: "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM
 * Serving on Commodity GPUs", technical summary, Methodology 1 ("Native
 * block-table decode engine") and 2 ("Calibrated adaptive policy").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers prefixed d_ are device pointers owned by the caller (the library
 *   never frees or keeps them).  Host pointers are read during the call only.
 * - fp16 means IEEE 754 binary16 (CUDA __half); buffers are passed as void*.
 * - Layouts (row-major, innermost last):
 *     q            [B][Hq][d]                    fp16
 *     k_cache      [num_pages][page_size][Hkv][d] fp16   ("NHD" pages)
 *     v_cache      [num_pages][page_size][Hkv][d] fp16
 *     block_table  [B][bt_stride]                int32  (physical page ids)
 *     seq_lens     [B]                           int32  (N*_i, real lengths)
 *     o            [B][Hq][d]                    fp16
 *     lse          [B][Hq]                       fp32   (natural log; may be NULL)
 *   Query head h reads KV head h / G with G = Hq / Hkv.  Token t of row i lives
 *   in page block_table[i][t / page_size], slot t % page_size.
 * - Every device buffer must be 16-byte aligned.
 * - `stream` is a cudaStream_t (CUstream) cast to void*; NULL is the legacy
 *   default stream.  Every call only enqueues work: none synchronizes, except
 *   pkv_get_error which says so.
 * - Return value: PKV_OK (0) or a negative status.  A failed call enqueues
 *   nothing.  pkv_last_error_string() gives a per-thread description of the
 *   last failure.  No C++ exception crosses this boundary.
 * - Supported shapes: d in {64, 128}; G = Hq/Hkv in [1, 8]; page_size a power
 *   of two in [8, 256]; split_tokens a positive multiple of page_size.  Other
 *   shapes return PKV_EUNSUPPORTED.
 * - Device-side checks (a block-table entry outside [0, num_pages), a length
 *   beyond the block table or the bucket, a workqueue larger than its
 *   capacity, a bounded wait that gave up) never fault or trap: the kernel
 *   records the first such event in the workspace's error word, replaces the
 *   offending page by zeros (or skips the work), and finishes.  Read it with
 *   pkv_get_error().
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_VERSION 2

/* status codes */
#define PKV_OK 0
#define PKV_EINVAL (-1)        /* bad argument: null/unaligned pointer, bad shape */
#define PKV_EUNSUPPORTED (-2)  /* valid but not implemented (see shapes above) */
#define PKV_ECUDA (-3)         /* a CUDA runtime/driver call failed */
#define PKV_EDEVICE (-4)       /* device-side check: bad page id or length */
#define PKV_ETIMEOUT (-5)      /* a bounded device wait gave up */
#define PKV_ECAPACITY (-6)     /* workqueue larger than max_tasks */

/* Execution paths (Methodology 2, "Calibrated adaptive policy"). */
typedef enum {
    PKV_PATH_BUCKETED_SPLIT = 0, /* rectangular B x Hkv x S_b grid over one length bucket */
    PKV_PATH_WORKQUEUE = 1,      /* compact 1D queue of non-empty (row, kv-head, split) tasks */
    PKV_PATH_SINGLE_PASS = 2     /* one task per (row, kv-head), no split, no merge */
} pkv_path_t;

/* A shape with B = 0 is accepted by every launching call, which then does
 * nothing and returns PKV_OK (its pointers are not examined). */
typedef struct {
    int32_t B;          /* batch rows, one query token each */
    int32_t Hq;         /* query heads */
    int32_t Hkv;        /* KV heads; Hq % Hkv == 0 */
    int32_t d;          /* head dim */
    int32_t page_size;  /* tokens per page (P) */
    int32_t num_pages;  /* pages in the pool (first dim of k_cache/v_cache) */
    int32_t bt_stride;  /* int32 elements between block-table rows */
    float scale;        /* score scale, normally 1/sqrt(d) */
} pkv_shape_t;

typedef struct {
    pkv_path_t path;
    int32_t split_tokens; /* C: tokens per split, a multiple of page_size
                             (ignored by PKV_PATH_SINGLE_PASS) */
    int32_t bucket_len;   /* BUCKETED_SPLIT: tokens covered by the grid,
                             S_b = ceil(bucket_len / C); 0 = bt_stride*page_size.
                             A row longer than the bucket is a device error. */
    int32_t max_tasks;    /* WORKQUEUE: task capacity of the workspace;
                             0 = Hkv * B * ceil(bt_stride*page_size / C) */
    int32_t merge;        /* split paths, for the step calls (pkv_decode_step
                             and its variants): PKV_MERGE_SEPARATE or
                             PKV_MERGE_FUSED (see pkv_decode_merge) */
    int32_t plan;         /* WORKQUEUE: PKV_PLAN_SEPARATE or
                             PKV_PLAN_IN_DECODE (see pkv_decode) */
} pkv_plan_cfg_t;

/* How a step combines the split states.  SEPARATE is the pages' structure
 * (Methodology 1, "Sequence splitting": a second kernel merges the states);
 * FUSED runs the same exact merge on the decode kernel's tail, one launch
 * fewer per step.  A zero-filled cfg selects SEPARATE. */
#define PKV_MERGE_SEPARATE 0
#define PKV_MERGE_FUSED 1

/* Where the workqueue's plan is built.  SEPARATE: the plan kernel (pkv_plan),
 * then the decode reads its task list.  IN_DECODE: for B <= PKV_SELF_PLAN_MAX_B
 * the decode kernel builds the same plan itself, so a step needs no plan
 * launch (pkv_decode documents it).  A zero-filled cfg selects SEPARATE. */
#define PKV_PLAN_SEPARATE 0
#define PKV_PLAN_IN_DECODE 1
#define PKV_SELF_PLAN_MAX_B 512

/* ---------------------------------------------------------------- sizes */

/* Bytes of the plan workspace: a 64-byte header (error word, task count, the
 * decode's task-claim and barrier counters), offsets[B+1] and, for WORKQUEUE,
 * the task list (16 bytes per task) followed by internal scheduling data (a
 * balance-ordered copy of the list and one int per row).  Every launching
 * entry point takes this workspace (it holds the error word).  Zero it once
 * after allocation: the header must start at zero; its counters are back at
 * zero after every launch and pkv_get_error() clears the error word. */
size_t pkv_plan_workspace_size(const pkv_shape_t *shape, const pkv_plan_cfg_t *cfg);

/* Bytes of the fp32 partial-state buffer for split paths: acc[slots][d] then
 * m[slots] then l[slots], where slots = B*S_b*Hq (BUCKETED_SPLIT) or
 * max_tasks*G (WORKQUEUE).  0 for SINGLE_PASS.  Slots are 32-bit indices: the
 * launching calls refuse a configuration with more than INT32_MAX of them
 * (PKV_EUNSUPPORTED). */
size_t pkv_partials_size(const pkv_shape_t *shape, const pkv_plan_cfg_t *cfg);

/* ----------------------------------------------------------- the path */

/* pkv_plan -- row-local bounds and the compact workqueue, built on the device
 * (Methodology 1, "Row-local bounds" and "Compact workqueue").
 * One kernel launch (a single CTA prefix scan) on `stream`:
 *   n_i = ceil(N*_i / C); offsets[i] = n_0 + ... + n_{i-1}; T = Hkv * sum n_i;
 *   tasks[k] = {i, g, j, state_base = (offsets[i] + j) * Hq + g * G} in
 *   lexicographic (row, kv-head, split) order; count = T.
 * The host never reads T back.  If T > max_tasks the count is set to 0 and
 * the error word to capacity; decode then does nothing and merge writes NaN.
 * For BUCKETED_SPLIT and SINGLE_PASS it is a no-op returning PKV_OK. */
int pkv_plan(const pkv_shape_t *shape, const pkv_plan_cfg_t *cfg,
             const int32_t *d_seq_lens, void *d_ws, void *stream);

/* pkv_decode -- split decode (Methodology 1, "Sequence splitting").
 * One kernel launch.  Every task (i, g, j) covers tokens
 * [j*C, min((j+1)*C, N*_i)) of row i and writes, for each of the G query heads
 * h of KV head g, the partial online-softmax state over s_t = scale * q_h.K_t:
 *   m = max_t s_t, l = sum_t exp(s_t - m), acc = sum_t exp(s_t - m) V_t (fp32)
 * into slot state_base + (h - g*G) of d_partials.  BUCKETED_SPLIT walks the
 * rectangular grid B x Hkv x S_b (state_base = (i*S_b + j)*Hq + g*G); an empty
 * split writes the neutral state (m=-inf, l=0, acc=0) and reads no KV.
 * WORKQUEUE walks the task list pkv_plan wrote into d_ws (enqueue pkv_plan
 * first on the same stream) -- unless cfg->plan == PKV_PLAN_IN_DECODE and
 * B <= PKV_SELF_PLAN_MAX_B: then every CTA derives the tasks from d_seq_lens
 * itself (prefix sums of each row's full and shorter splits, in shared
 * memory) and the launch also writes into d_ws the plan pkv_plan would have
 * written (header, offsets, task list), so pkv_merge follows as usual and no
 * pkv_plan is needed.  K/V pages are read in place through the block table;
 * no page is repacked. */
int pkv_decode(const pkv_shape_t *shape, const pkv_plan_cfg_t *cfg, void *d_ws,
               const void *d_q, const void *d_k_cache, const void *d_v_cache,
               const int32_t *d_block_table, const int32_t *d_seq_lens,
               float *d_partials, void *stream);

/* pkv_merge -- exact log-sum-exp merge (Methodology 1, "Sequence splitting":
 * a separate merge kernel combines the split states exactly).
 * One kernel launch.  For each (row i, query head h) it reads the n_i =
 * ceil(N*_i / C) states of that row only (row-local bounds) and writes
 *   M = max_j m_j, L = sum_j l_j exp(m_j - M),
 *   o[i][h] = sum_j acc_j exp(m_j - M) / L  (fp16, round to nearest),
 *   lse[i][h] = M + ln L                    (fp32, if lse != NULL).
 * A row with N*_i = 0 gets o = 0 and lse = -inf. */
int pkv_merge(const pkv_shape_t *shape, const pkv_plan_cfg_t *cfg, void *d_ws,
              const int32_t *d_seq_lens, const float *d_partials,
              void *d_o, float *d_lse, void *stream);

/* pkv_single_pass -- the no-split route of the policy (Methodology 2: the
 * route the pages hand to an external single-kernel library; here our own
 * kernel).  One kernel launch; one task per (row, kv-head) over the whole row,
 * writing o and lse directly as pkv_merge would. */
int pkv_single_pass(const pkv_shape_t *shape, void *d_ws,
                    const void *d_q, const void *d_k_cache, const void *d_v_cache,
                    const int32_t *d_block_table, const int32_t *d_seq_lens,
                    void *d_o, float *d_lse, void *stream);

/* pkv_decode_merge -- pkv_decode with the exact merge of pkv_merge on its
 * tail (cfg->merge is not consulted, nor cfg->plan: on the workqueue enqueue
 * pkv_plan first).  One kernel launch.  Every split writes
 * its state as pkv_decode does; the kernel's CTAs then meet at a grid-wide
 * barrier (counters in d_ws; every CTA is resident at once, and the wait is
 * bounded: a CTA that gives up reports PKV_ETIMEOUT) and share out the
 * (row, query head) merges, computed with pkv_merge's formulas.  A row with
 * one split writes o / lse directly; a row with N*_i = 0 gets o = 0,
 * lse = -inf; a workqueue overflow writes NaN as pkv_merge does.  Results
 * equal pkv_decode + pkv_merge up to the order of the fp32 sums.  Launches on
 * one workspace must not overlap on the GPU.  The barrier needs the whole grid
 * (at most the CTAs the GPU holds at once) resident together: kernels of other
 * streams that keep SMs busy delay it, and if it cannot fill within 1 s the
 * CTAs give up and report PKV_ETIMEOUT rather than wait on. */
int pkv_decode_merge(const pkv_shape_t *shape, const pkv_plan_cfg_t *cfg, void *d_ws,
                     const void *d_q, const void *d_k_cache, const void *d_v_cache,
                     const int32_t *d_block_table, const int32_t *d_seq_lens,
                     float *d_partials, void *d_o, float *d_lse, void *stream);

/* pkv_decode_step -- one whole decode step on the path cfg->path:
 * WORKQUEUE = pkv_plan + pkv_decode + pkv_merge, BUCKETED_SPLIT = pkv_decode +
 * pkv_merge, SINGLE_PASS = pkv_single_pass; with cfg->merge == PKV_MERGE_FUSED
 * pkv_decode_merge replaces pkv_decode + pkv_merge.  WORKQUEUE with
 * cfg->plan == PKV_PLAN_IN_DECODE, the separate merge and
 * B <= PKV_SELF_PLAN_MAX_B drops the pkv_plan launch (the decode plans for
 * itself); otherwise the field has no effect.  Same arguments and errors as
 * those calls; d_partials may be NULL for SINGLE_PASS. */
int pkv_decode_step(const pkv_shape_t *shape, const pkv_plan_cfg_t *cfg, void *d_ws,
                    const void *d_q, const void *d_k_cache, const void *d_v_cache,
                    const int32_t *d_block_table, const int32_t *d_seq_lens,
                    float *d_partials, void *d_o, float *d_lse, void *stream);

/* pkv_decode_step_host -- one decode step with the step's inputs and outputs in
 * host memory, for a serving loop that keeps the KV cache resident on the
 * device: copies h_q into d_q (and, when non-NULL, h_block_table into
 * d_block_table and h_seq_lens into d_seq_lens) on `stream`, runs
 * pkv_decode_step, copies d_o into h_o (and d_lse into h_lse when both are
 * non-NULL), then synchronizes `stream`.  One cudaMemcpyAsync per buffer --
 * except that a page-locked (pinned or registered), 16-byte aligned host
 * buffer is used in place: h_q, h_block_table and h_seq_lens are then read by
 * the step's kernels, h_o and h_lse written by its last kernel, and the
 * matching device buffer is not written.  Pageable host buffers go through the
 * device buffers (their copies are then synchronous with the host).  All
 * arguments are checked before anything is enqueued.  Same path semantics,
 * layouts and errors as pkv_decode_step. */
int pkv_decode_step_host(const pkv_shape_t *shape, const pkv_plan_cfg_t *cfg, void *d_ws,
                         float *d_partials, const void *h_q, void *d_q,
                         const int32_t *h_block_table, int32_t *d_block_table,
                         const int32_t *h_seq_lens, int32_t *d_seq_lens,
                         const void *d_k_cache, const void *d_v_cache,
                         void *d_o, void *h_o, float *d_lse, float *h_lse, void *stream);

/* pkv_append_decode_step_host -- one step of a serving loop that grows every
 * row by one token, with the step's inputs and outputs in host memory and the
 * KV cache, block table and lengths resident on the device (they are state the
 * step advances).  (Not a step of the pages' method by itself: the serving
 * loop around it, whose wall clock the pages' evaluation protocol,
 * Methodology 3, counts with the host's share.)  In order, on `stream`:
 *   1. copies h_q [B][Hq][d] into d_q and the new token's h_k_new, h_v_new
 *      [B][Hkv][d] (fp16) into d_k_new, d_v_new -- one cudaMemcpyAsync each,
 *      except that a page-locked (pinned or registered), 16-byte aligned h_q
 *      is read in place by the decode, and page-locked h_k_new and h_v_new by
 *      the append, and then d_q (d_k_new, d_v_new) is not written;
 *   2. WORKQUEUE: pkv_append_plan (appends, allocates pages from the device
 *      free list when d_free_pages != NULL, and plans unless the decode will),
 *      then pkv_decode + pkv_merge (pkv_decode_merge with PKV_MERGE_FUSED),
 *      all with `cfg`; other paths: pkv_append, then pkv_decode_step;
 *   3. copies d_o into h_o (and d_lse into h_lse when both are non-NULL) --
 *      except that a page-locked, 16-byte aligned h_o (h_lse) is written
 *      straight by the step's last kernel and d_o (d_lse) is then not written;
 *   4. synchronizes `stream`.
 * After the call every row has one more token and o / lse are those of the
 * advanced lengths.  Page-locked host buffers save the copies above; pageable
 * ones work too (their copies are then synchronous with the host).  The device
 * buffers d_q, d_k_new, d_v_new and d_o are always required.  d_free_pages / d_free_count go together and only with the
 * WORKQUEUE path.  All arguments are checked before anything is enqueued;
 * device-side results (a row without room, an exhausted free list, a bad page
 * id) land in the error word as for those calls (read with pkv_get_error). */
int pkv_append_decode_step_host(const pkv_shape_t *shape, const pkv_plan_cfg_t *cfg, void *d_ws,
                                float *d_partials, const void *h_q, void *d_q,
                                const void *h_k_new, const void *h_v_new, void *d_k_new,
                                void *d_v_new, int32_t *d_block_table, int32_t *d_seq_lens,
                                const int32_t *d_free_pages, int32_t *d_free_count,
                                void *d_k_cache, void *d_v_cache, void *d_o, void *h_o,
                                float *d_lse, float *h_lse, void *stream);

/* pkv_append_plan --the step's KV write fused into the workqueue plan: one
 * kernel launch that appends one token per row exactly as pkv_append does and
 * then builds pkv_plan's task list from the advanced lengths.  With
 * d_free_pages != NULL a token that starts a new page (N % page_size == 0)
 * takes a page from the device free list d_free_pages[0 .. *d_free_count)
 * (the top of the stack is the end): rows needing one are served in row order
 * from the top, block_table[i][N / page_size] is set to it and *d_free_count
 * drops by the pages taken.  A row with no free page left, no room in its
 * block table or a bad page id keeps its length and the error word records it.
 * cfg->path must be WORKQUEUE.  With cfg->plan == PKV_PLAN_IN_DECODE, the
 * separate merge and B <= PKV_SELF_PLAN_MAX_B the decode that follows builds
 * the plan itself (see pkv_decode): the launch then only appends and
 * allocates -- same rule, same results, one CTA per row -- writes no plan,
 * and counts as an append launch in pkv_get_counters.  (Not a step of the
 * pages' method: the per-step KV write and page allocation of a serving loop,
 * folded into the launch the workqueue path makes anyway.) */
int pkv_append_plan(const pkv_shape_t *shape, const pkv_plan_cfg_t *cfg, void *d_ws,
                    const void *d_k_new, const void *d_v_new, int32_t *d_block_table,
                    int32_t *d_seq_lens, const int32_t *d_free_pages, int32_t *d_free_count,
                    void *d_k_cache, void *d_v_cache, void *stream);

/* pkv_append -- write one new token per row into the paged cache.
 * (Not a step of the pages' method: the per-step KV write of a serving loop.)
 * One kernel launch.  For every row i with N = seq_lens[i]: copies
 * k_new[i][g][:], v_new[i][g][:] ([B][Hkv][d] fp16) into page
 * block_table[i][N / page_size], slot N % page_size, then sets
 * seq_lens[i] = N + 1 in place.  The block table must already name that page.
 * A row whose next slot is beyond the block table or whose page id is out of
 * range is left unchanged and recorded in the error word. */
int pkv_append(const pkv_shape_t *shape, void *d_ws, const void *d_k_new,
               const void *d_v_new, const int32_t *d_block_table, int32_t *d_seq_lens,
               void *d_k_cache, void *d_v_cache, void *stream);

/* pkv_decode_step_rows -- the launch group of the exact-length-bucket scheme
 * (Results, "Scheduling overhead": the scheme the compact workqueue replaces
 * launches one group per exact row length): pkv_decode + pkv_merge on the
 * BUCKETED_SPLIT path over the rows d_rows[0..n_rows) of the batch only
 * (distinct indices in [0, B); an entry outside is a device error and that
 * row is skipped).  bucket_len must cover the group's longest row; d_partials
 * holds n_rows*S_b*Hq states (pkv_partials_size with B = n_rows).  Two kernel
 * launches (one with PKV_MERGE_FUSED); o and lse rows outside the list are
 * left untouched. */
int pkv_decode_step_rows(const pkv_shape_t *shape, const pkv_plan_cfg_t *cfg, void *d_ws,
                         const int32_t *d_rows, int32_t n_rows,
                         const void *d_q, const void *d_k_cache, const void *d_v_cache,
                         const int32_t *d_block_table, const int32_t *d_seq_lens,
                         float *d_partials, void *d_o, float *d_lse, void *stream);

/* pkv_exact_length_groups -- the launch groups of the exact-length-bucket
 * scheme (Results, "Scheduling overhead": the scheme the compact workqueue
 * replaces launches one split + merge pair per distinct row length), computed
 * on the host from the host lengths seq_lens[B]; no CUDA call.  Writes:
 *   rows[0 .. B): the rows with tokens grouped by length -- lengths ascending,
 *     rows ascending within a length -- then the rows of length 0;
 *   group_start[0 .. n_groups]: group g is rows[group_start[g] ..
 *     group_start[g + 1]), group_start[n_groups] = the rows with tokens;
 *   group_len[0 .. n_groups): the length of group g;
 *   *n_groups: the number of distinct non-zero lengths.
 * Arrays hold B (rows, group_len) and B + 1 (group_start) entries.  Each group
 * runs as pkv_decode_step_rows with bucket_len = its length; the rows of length
 * 0, if any, as one more pkv_decode_step_rows (any bucket_len), which gives them
 * o = 0 and lse = -inf.  A negative length is PKV_EINVAL. */
int pkv_exact_length_groups(const int32_t *seq_lens, int32_t B, int32_t *rows,
                            int32_t *group_start, int32_t *group_len, int32_t *n_groups);

/* pkv_decode_step_noalloc -- pkv_decode_step for callers that cannot
 * allocate device memory.  No counterpart in the paper: it serves callers that
 * must not call cudaMalloc -- code running inside an allocator's callbacks,
 * plugins of runtimes that own every device allocation, paths that must avoid
 * the allocator's implicit synchronisation -- and so cannot supply the plan
 * workspace and partial-state buffers.  The caller passes inputs and outputs
 * as for pkv_decode_step; the scratch is a file-scope device array of
 * PKV_NOALLOC_SCRATCH_BYTES that every GPU loading libpkv holds until the
 * process exits.  The call allocates nothing.
 * - A step whose plan workspace (rounded up to 256 bytes) plus partial states
 *   exceed PKV_NOALLOC_SCRATCH_BYTES is rejected with PKV_ECAPACITY.
 * - Set-up on first use: the first call on each device looks up the array's
 *   device address (with that device current).  Under CUDA's default lazy
 *   module loading that first call -- and the first call of each path, merge
 *   and plan mode, whose kernels then load -- also brings the library's code
 *   and the array onto the device, which the CUDA driver backs with device
 *   memory.  So make one call per configuration you will use outside any
 *   context where allocation is forbidden, and before any stream capture (or
 *   run with CUDA_MODULE_LOADING=EAGER); later calls allocate nothing.
 * - Every call shares the one array and it keeps the last call's contents:
 *   the call clears the workspace header (error word, task count, counters),
 *   but calls that overlap on the GPU (different streams, or other host
 *   threads) race -- serialize them.  Device-side check results stay in the array and are not
 *   reported; callers needing pkv_get_error use pkv_decode_step. */
#define PKV_NOALLOC_SCRATCH_BYTES (16 * 1024 * 1024)

int pkv_decode_step_noalloc(const pkv_shape_t *shape, const pkv_plan_cfg_t *cfg,
                            const void *d_q, const void *d_k_cache, const void *d_v_cache,
                            const int32_t *d_block_table, const int32_t *d_seq_lens,
                            void *d_o, float *d_lse, void *stream);

/* ------------------------------------------------------------- policy */

/* Thresholds of the calibrated policy (Methodology 2).  The pages route
 * B = 1 long-context to the length-bucketed split, B >= 8 long-context to the
 * compact workqueue and everything else (including B = 4) to a single-kernel
 * path; what counts as "long" and the batch cut-offs are calibrated.  Here
 * each split route has its own long-context cut-off:
 *   B <= bucketed_max_batch  and N_max >= bucketed_min_tokens  -> BUCKETED_SPLIT
 *   else B >= workqueue_min_batch and N_max >= workqueue_min_tokens -> WORKQUEUE
 *   else SINGLE_PASS.
 * The workqueue's split size grows with the batch, because every split writes
 * a partial state: C starts at split_tokens and doubles while
 * B * ceil(N_max / C) > workqueue_target_splits and the longest row would keep
 * at least workqueue_min_long_splits splits (ceil(N_max / 2C) of them), up to
 * workqueue_max_split_tokens (a target of 0 keeps C = split_tokens). */
typedef struct {
    int32_t bucketed_min_tokens;   /* long-context cut-off of the bucketed route */
    int32_t bucketed_max_batch;    /* largest B routed to BUCKETED_SPLIT */
    int32_t workqueue_min_tokens;  /* long-context cut-off of the workqueue route */
    int32_t workqueue_min_batch;   /* smallest B routed to WORKQUEUE */
    int32_t split_tokens;          /* smallest C handed to WORKQUEUE */
    int32_t bucketed_split_tokens; /* C handed to BUCKETED_SPLIT */
    int32_t workqueue_max_split_tokens; /* largest C handed to WORKQUEUE */
    int32_t workqueue_target_splits;    /* (row, split) pairs the workqueue's C aims at */
    int32_t workqueue_min_long_splits;  /* splits the longest row keeps as C grows */
} pkv_policy_cfg_t;

/* Fill `cfg` with the thresholds calibrated on GB300 (calibration seed
 * 20260622, checked on held-out seed 20260623). */
void pkv_policy_default(pkv_policy_cfg_t *cfg);

/* Choose the path for a batch of B rows whose longest row has n_max tokens.
 * cfg may be NULL (defaults).  Host only, deterministic, no CUDA call. */
int pkv_policy(int32_t B, int32_t n_max, const pkv_policy_cfg_t *cfg,
               pkv_path_t *out_path, int32_t *out_split_tokens);

/* Learned cost model (technical summary, Significance: the authors name a
 * learned cost model for the thresholds as future work).  For route r
 * (a path and a split size) log(t_r) = w_r . f with
 *   f = [1, lb, ln, ls, lb*ln, lb^2, ln^2, fill, fill*lb, ls^2],
 *   lb = log2 B, ln = log2 N_max, ls = log2 max(N_sum, 1), fill = N_sum / (B N_max),
 * N_sum being the batch's total tokens.  Defaults are fitted by least squares
 * on GB300 step times of the calibration seed (paged_kv_gqa_09_gb300/calibrate.py). */
#define PKV_COST_FEATURES 10
#define PKV_COST_MAX_ROUTES 16

typedef struct {
    int32_t path;          /* a pkv_path_t */
    int32_t split_tokens;  /* C of the route (ignored by SINGLE_PASS) */
    float w[PKV_COST_FEATURES];
} pkv_cost_route_t;

typedef struct {
    int32_t n_routes;
    pkv_cost_route_t route[PKV_COST_MAX_ROUTES];
} pkv_cost_model_t;

/* Fill `model` with the GB300-fitted routes. */
void pkv_cost_model_default(pkv_cost_model_t *model);

/* Pick the route of smallest predicted step time for B rows with longest
 * row n_max and total tokens n_sum (host only, deterministic).  model may be
 * NULL (defaults).  B = 0 or n_max = 0 gives SINGLE_PASS. */
int pkv_policy_learned(int32_t B, int32_t n_max, int64_t n_sum, const pkv_cost_model_t *model,
                       pkv_path_t *out_path, int32_t *out_split_tokens);

/* ----------------------------------------------------------- counters */

/* Scheduler-derived counters (technical summary, Methodology 3 and Results,
 * "Scheduling overhead").  pkv_get_counters returns what the library actually
 * launched since the last pkv_reset_counters (process-wide, thread-safe). */
typedef struct {
    int64_t plan_launches;
    int64_t decode_launches;
    int64_t merge_launches;
    int64_t single_pass_launches;
    int64_t append_launches;
} pkv_counters_t;

int pkv_get_counters(pkv_counters_t *out);
int pkv_reset_counters(void);

/* Model of one decode step, computed on the host from the real lengths
 * (host array seq_lens[B]):
 *   attn_launches: kernel launches of the attention path (split + merge, or
 *     the single pass; the plan launch is counted apart in plan_launches);
 *     for exact-length buckets, one split and one merge per distinct length;
 *   tasks: non-empty (row, kv-head, split) tasks; grid_tasks: tasks in the
 *     launched grid including empty rectangular cells;
 *   merge_state_bytes: fp32 state bytes written by the split kernel plus
 *     read by the merge, (d + 2) * 4 per state;
 *   kv_bytes: sum_i N*_i * Hkv * d * 2 * 2.
 * path_or_exact: a pkv_path_t, or 3 for exact-length buckets. */
typedef struct {
    int64_t attn_launches;
    int64_t plan_launches;
    int64_t tasks;
    int64_t grid_tasks;
    int64_t states_written;
    int64_t states_read;
    int64_t merge_state_bytes;
    int64_t kv_bytes;
} pkv_step_model_t;

int pkv_step_model(int32_t path_or_exact, const pkv_shape_t *shape, int32_t split_tokens,
                   int32_t bucket_len, const int32_t *seq_lens, pkv_step_model_t *out);

/* ------------------------------------------------------------- errors */

/* Synchronizes `stream`, reads and clears the device error word in d_ws and
 * returns PKV_OK, PKV_EDEVICE, PKV_ETIMEOUT or PKV_ECAPACITY (detail in
 * pkv_last_error_string()). */
int pkv_get_error(void *d_ws, void *stream);

/* Test hook for the bounded-wait path: the next n decode or single-pass
 * launches run with CTA 0 leaving its first pipeline stage unfilled, so the
 * consumer warps' wait on it runs out (after about 1 s); the kernel records
 * PKV_ETIMEOUT, drains its own copies and returns.  Nothing faults, traps or
 * hangs; the outputs of such a launch are meaningless.  0 switches it off.
 * The hook is off unless the process runs with the environment variable
 * PKV_TEST_HOOKS=1 (read at each call); otherwise it changes nothing and
 * returns PKV_EUNSUPPORTED.  It stays in the one library so that the tests
 * exercise the very binary a serving process loads. */
int pkv_test_starve_next_decodes(int32_t n);

/* Description of the last failure on the calling thread ("" if none). */
const char *pkv_last_error_string(void);

/* PKV_VERSION of the loaded library. */
int pkv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
