/*
 * nanospec.h — C ABI of the dynamic-vocabulary draft LM head (GB300, sm_103a).
 *
 * The library keeps, per sequence, the candidate stream of the NanoSpec /
 * MicroSpec method resident on the GPU, turns it into the active vocabulary
 * I_t with a bitmap, packs W_head[I_t, :] into a contiguous buffer and
 * projects draft hidden states through that sub-head, returning top-k token
 * ids in the global vocabulary.
 *
 * Sources (the paper appears as NanoSpec on one page and as MicroSpec on
 * another; section numbers are MicroSpec's):
 *   MicroSpec §3.1 Eq. 1                 z_t = W_head h_t
 *   MicroSpec §3.2 stream-init equation  S_init = x_{1:L} (+) tuple(U_i T_Kpre(z_i))
 *   MicroSpec §3.2 stream-update eq.     S_new = S_old (+) tuple(C_draft) (+) tuple(C_ver)
 *   MicroSpec §3.2 sliding-window eq.    I_{t+1} = Unique(Suffix(S_new, W_max))
 *   MicroSpec §3.3 "Avoiding Sparse Computation via Asynchronous Gathering"
 *   MicroSpec §3.3 "Eliminating Overhead via GPU-Resident State Management"
 *
 * Conventions for every call:
 *   - Token ids are 0-based int32 in [0, V).
 *   - bf16 tensors are passed as uint16_t bit patterns, row-major.
 *   - Pointers named d_* are DEVICE pointers on the current CUDA device; the
 *     caller owns them and they are only borrowed for the duration of the
 *     work the call enqueues.  W_head must stay valid while work that reads
 *     it is in flight.
 *   - ns_stream is a cudaStream_t, ns_event a cudaEvent_t (NULL = legacy
 *     default stream / no event).
 *   - All calls are asynchronous on the given stream.  No call synchronises
 *     the host except ns_get_error, ns_create and ns_destroy.  |I_t| stays on
 *     the device; kernels size themselves from W_max and read the count.
 *   - A call returns NS_ERR_ARG, without enqueuing anything, when an
 *     argument is invalid; NS_ERR_CUDA when a CUDA call fails.
 *   - Device-side problems (an input id outside [0, V)) do not stop the
 *     stream: the offending entry is skipped and a sticky flag is set, read by
 *     ns_get_error.
 *   - Work for one sequence must be ordered (one stream, or events).  Work
 *     for different sequences may run concurrently.
 *   - Every Top-K and top-k orders by value, larger first, ties to the
 *     smaller id; -0.0 ties +0.0; +inf and -inf are ordered like any value;
 *     NaN never ranks (a row with fewer than K non-NaN values yields fewer
 *     entries, see the calls).
 */
#ifndef NANOSPEC_H
#define NANOSPEC_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Entry points are exported even when the library is built with hidden
 * default visibility. */
#if defined(__GNUC__)
#define NS_API __attribute__((visibility("default")))
#else
#define NS_API
#endif

typedef int32_t ns_status;
#define NS_OK 0
#define NS_ERR_ARG (-1)     /* invalid argument; nothing enqueued            */
#define NS_ERR_CUDA (-2)    /* a CUDA runtime call or launch failed          */
#define NS_ERR_OOM (-3)     /* device allocation failed                      */
#define NS_ERR_TIMEOUT (-4) /* a bounded device-side wait ran out            */
#define NS_ERR_STATE (-5)   /* call out of order (e.g. append before init)   */

/* Sticky device error flags (bit mask), read with ns_get_error. */
#define NS_FLAG_BAD_ID 0x1u    /* an input token id outside [0, V) was skipped */
#define NS_FLAG_OVERFLOW 0x2u  /* an internal capacity was exceeded (bug)      */
#define NS_FLAG_TIMEOUT 0x4u   /* a bounded device-side wait gave up            */
#define NS_FLAG_INTERNAL 0x8u  /* an internal id was out of range and skipped (a bug); bits 8..15 name the site */

typedef void *ns_stream; /* cudaStream_t */
typedef void *ns_event;  /* cudaEvent_t  */

/* Limits of the library. */
#define NS_MAX_SELECT_K 16 /* K_pre and K_ver                               */
#define NS_MAX_TOPK 32     /* k of the sub-head top-k                       */
#define NS_MAX_ROWS 64     /* hidden rows per projection call (draft nodes) */

typedef struct ns_config {
  int32_t V;          /* vocabulary size (rows of W_head), >= 1               */
  int32_t H;          /* hidden size d (columns of W_head), multiple of 64    */
  int32_t W_max;      /* sliding-window length, >= 1                          */
  int32_t K_pre;      /* Top-K per prefill row, 0..NS_MAX_SELECT_K            */
  int32_t K_ver;      /* Top-K of the verify row, 0..NS_MAX_SELECT_K          */
  int32_t max_tree;   /* most draft-tree ids per append, 0..NS_MAX_ROWS       */
  int32_t max_k;      /* most top-k per hidden row, 1..NS_MAX_TOPK            */
  int32_t batch;      /* independent sequences, >= 1                          */
  int32_t max_prompt; /* longest prompt accepted by ns_stream_init, >= 1      */
} ns_config;

typedef struct ns_handle ns_handle;

/* Returns a static, human-readable name of a status code. */
NS_API const char *ns_status_string(ns_status s);

/*
 * Allocates all device state for cfg->batch sequences on the current device
 * (per sequence: ring of W_max int32 stream entries, V occurrence counts,
 * ceil(V/32) bitmap words, I_t as W_max int32 + count, the packed sub-head
 * W_max x H bf16 — MicroSpec §3.3's pre-allocated contiguous buffer — and
 * scratch).  The state starts empty; every sequence must be initialised with
 * ns_stream_init before it is appended to.  Synchronises the device.
 * *out receives the handle; NS_ERR_ARG on bad limits, NS_ERR_OOM when
 * allocation fails.
 */
NS_API ns_status ns_create(const ns_config *cfg, ns_handle **out);

/* Synchronises the device and frees everything the handle owns. */
NS_API ns_status ns_destroy(ns_handle *h);

/* Bytes of device memory the handle holds (all sequences). */
NS_API int64_t ns_device_bytes(const ns_handle *h);

/*
 * Prefill: S_init = prompt (+) tuple(union over i of T_Kpre(z_i))
 * (MicroSpec §3.2, stream-initialisation equation).
 *   d_prompt          int32 [L], 0 <= L <= max_prompt, ids in [0, V); L = 0
 *                     (d_prompt may then be NULL) starts an empty stream, so
 *                     the vocabulary comes from decode-time candidates alone
 *                     (the Ext-only ablation of NanoSpec's evaluation)
 *   d_prefill_logits  fp32 [L x V] row-major, row i = z_i (may be NULL when
 *                     K_pre == 0 or L == 0)
 * The union is deduplicated in first-occurrence order, position-major then
 * rank-minor (largest logit first, ties to the smaller id); prompt ids are
 * kept verbatim.  Only the last W_max entries of S_init are stored.  Resets
 * the sequence's previous state.  Out-of-range prompt ids are skipped and
 * flag NS_FLAG_BAD_ID.  Leaves I_t unbuilt (call ns_build_active_vocab).
 */
NS_API ns_status ns_stream_init(ns_handle *h, int32_t seq, const int32_t *d_prompt, int32_t L,
                         const float *d_prefill_logits, ns_stream stream);

/*
 * Decode-step update S_new = S_old (+) tuple(C_draft) (+) tuple(C_ver)
 * (MicroSpec §3.2, "Dynamic Stream Update" and the stream-update equation),
 * then the window counts and bitmap of Unique(Suffix(S_new, W_max)).
 *   d_tree_ids       int32 [n_tree], 0 <= n_tree <= max_tree: every node of
 *                    the draft tree; C_draft = distinct ids in first-occurrence
 *                    node order (out-of-range ids skipped, NS_FLAG_BAD_ID)
 *   d_verify_logits  fp32 [n_verify x V] row-major; C_ver = T_Kver of row
 *                    verify_row (value descending, ties to the smaller id).
 *                    May be NULL when K_ver == 0.
 * Everything appended refreshes recency; entries older than the last W_max
 * are evicted.  Does not rebuild I_t.
 */
NS_API ns_status ns_stream_append(ns_handle *h, int32_t seq, const int32_t *d_tree_ids, int32_t n_tree,
                           const float *d_verify_logits, int32_t n_verify, int32_t verify_row,
                           ns_stream stream);

/*
 * I_t = Unique(Suffix(S, W_max)) read out of the bitmap in ascending id order
 * (MicroSpec §3.2 sliding-window equation; §3.3 GPU-resident bitmaps).
 * Writes the device list and its device count (see ns_get_active).
 */
NS_API ns_status ns_build_active_vocab(ns_handle *h, int32_t seq, ns_stream stream);

/*
 * packed[j, :] = W_head[I_t[j], :] for j < |I_t| (MicroSpec §3.3, gathering
 * into the pre-allocated contiguous buffer).  Meant for a copy stream that
 * overlaps the draft backbone: when `done` is not NULL it is recorded on
 * copy_stream after the gather, and the projection's stream should wait on
 * it.  d_W_head: bf16 [V x H] row-major.
 */
NS_API ns_status ns_gather_head_rows(ns_handle *h, int32_t seq, const uint16_t *d_W_head,
                              ns_stream copy_stream, ns_event done);

/*
 * Sub-head projection and top-k on the packed buffer:
 *   logits[r, j] = sum_h hidden[r, h] * packed[j, h]   (Eq. 1 on W_head[I_t,:]),
 * bf16 inputs, fp32 accumulation, for r < n, j < |I_t|; then per row the k
 * largest logits (ties to the smaller id) mapped to global ids I_t[j].
 *   d_hidden     bf16 [n x H], 1 <= n <= NS_MAX_ROWS
 *   k            1 <= k <= max_k
 *   d_logits     fp32 [n x ld_logits] or NULL; columns >= |I_t| untouched;
 *                ld_logits >= W_max
 *   d_topk_ids   int32 [n x k]; rows with |I_t| < k are padded with -1
 *   d_topk_vals  fp32  [n x k]; padding is -inf
 */
NS_API ns_status ns_sub_lm_head_logits_topk(ns_handle *h, int32_t seq, const uint16_t *d_hidden, int32_t n,
                                     int32_t k, float *d_logits, int32_t ld_logits,
                                     int32_t *d_topk_ids, float *d_topk_vals, ns_stream stream);

/*
 * One whole decode step for one sequence, in as few launches as the library
 * can: ns_stream_append, ns_build_active_vocab, the gather (writing the
 * packed buffer) and the projection with top-k, with the same arguments and
 * results as those calls made in order on `stream`.  Where the device holds
 * the whole grid at once it is ONE cooperative launch (ns_step_launches
 * returns 1): while some warps of every CTA update the window (a slice of
 * the verify row each, a grid barrier, the merge, append, evict, compact),
 * the others already project the rows of I_{t-1} and of the tree ids, and
 * each column is written at its id's position once I_t is known; a second
 * grid barrier precedes the per-row top-k.  When the window changed since
 * I_t was last built (ns_stream_init or ns_stream_append without
 * ns_build_active_vocab) the same launch projects I_t after computing it
 * (same results, slower).  Otherwise it is ns_state_update followed by
 * ns_gather_sub_lm_head_topk.
 */
NS_API ns_status ns_step(ns_handle *h, int32_t seq, const int32_t *d_tree_ids, int32_t n_tree,
                  const float *d_verify_logits, int32_t n_verify, int32_t verify_row,
                  const uint16_t *d_W_head, const uint16_t *d_hidden, int32_t n, int32_t k,
                  float *d_logits, int32_t ld_logits, int32_t *d_topk_ids, float *d_topk_vals,
                  ns_stream stream);

/* Kernel launches one ns_step makes on this handle (1 or 2; 0 for NULL). */
NS_API int32_t ns_step_launches(const ns_handle *h);

/*
 * One decode step for sequences 0 .. n_seq-1 of the handle together (batched
 * serving: independent streams, bitmaps and buffers), in two launches per 32
 * sequences: the state updates of all of them (one cluster each), then one
 * fused gather + projection + top-k over all their tiles (the grouped
 * projection n_seq x [n x H] . [|I_t^b| x H]^T).  Results equal n_seq calls of
 * ns_step, one per sequence, in order:
 *   d_tree_ids       int32 [n_seq x n_tree]       sequence b's tree ids in row b
 *   d_verify_logits  fp32  [n_seq x n_verify x V] sequence b's verify block
 *   verify_rows      HOST int32 [n_seq]           the row of each block to rank
 *   d_hidden         bf16  [n_seq x n x H]
 *   d_logits         fp32  [n_seq x n x ld_logits] or NULL
 *   d_topk_ids/vals        [n_seq x n x k]
 * Every sequence must have been initialised (NS_ERR_STATE otherwise).
 */
NS_API ns_status ns_step_batch(ns_handle *h, int32_t n_seq, const int32_t *d_tree_ids, int32_t n_tree,
                               const float *d_verify_logits, int32_t n_verify, const int32_t *verify_rows,
                               const uint16_t *d_W_head, const uint16_t *d_hidden, int32_t n, int32_t k,
                               float *d_logits, int32_t ld_logits, int32_t *d_topk_ids, float *d_topk_vals,
                               ns_stream stream);

/*
 * One decode step for sequences 0 .. n_seq-1 with ONE gather for all of them
 * (the batched reading of MicroSpec §3.3's gathering into a contiguous
 * buffer; the pages serve one sequence): every sequence's state update as in
 * ns_step_batch, then U = the union of their active vocabularies in
 * ascending id order (an OR of their window bitmaps, compacted), one gather
 * of W_head[U, :] into the handle's union buffer, and every sequence's
 * hidden rows projected through all of U, each sequence ranking only the
 * columns of its own I_t (its window bitmap is the mask).  A row of W_head
 * that several sequences hold crosses HBM once.  Results:
 *   d_logits    fp32 [n_seq x n x ld_logits] or NULL, ld_logits >= the union
 *               capacity (ns_get_union): sequence b's logits over all of U,
 *               column j <-> U[j], columns >= |U| untouched
 *   d_topk_ids/vals  [n_seq x n x k]: as ns_step_batch (each sequence's top-k
 *               over its own I_t; equal to ns_step_batch's up to rounding)
 * Other arguments as ns_step_batch.  The handle must hold more than one
 * sequence (NS_ERR_STATE otherwise: it has no union buffers).
 */
NS_API ns_status ns_step_batch_union(ns_handle *h, int32_t n_seq, const int32_t *d_tree_ids, int32_t n_tree,
                                     const float *d_verify_logits, int32_t n_verify, const int32_t *verify_rows,
                                     const uint16_t *d_W_head, const uint16_t *d_hidden, int32_t n, int32_t k,
                                     float *d_logits, int32_t ld_logits, int32_t *d_topk_ids, float *d_topk_vals,
                                     ns_stream stream);

/*
 * Device pointers to the union of the last ns_step_batch_union (owned by the
 * handle; NS_ERR_STATE for a handle of one sequence).  Any out-pointer may be
 * NULL.
 *   ids       int32 [capacity]   U ascending (first *count valid)
 *   count     int32 [1]          |U|
 *   bitmap    uint32 [ceil(V/32)] bit i set iff i in U
 *   packed    bf16 [capacity x H] rows j < |U| = W_head[U[j], :]
 *   capacity  HOST int64: min(batch x W_max, V)
 */
NS_API ns_status ns_get_union(ns_handle *h, const int32_t **ids, const int32_t **count, const uint32_t **bitmap,
                              const uint16_t **packed, int64_t *capacity);

/*
 * The state half of ns_step in one launch: ns_stream_append followed by
 * ns_build_active_vocab (the "GPU-resident state update" that determines
 * I_{t+1}, MicroSpec §3.3).  Arguments as ns_stream_append.
 */
NS_API ns_status ns_state_update(ns_handle *h, int32_t seq, const int32_t *d_tree_ids, int32_t n_tree,
                                 const float *d_verify_logits, int32_t n_verify, int32_t verify_row,
                                 ns_stream stream);

/*
 * The sub-head half of ns_step: the gather of W_head[I_t, :] into the packed
 * buffer fused with the projection (each row is read from HBM once, written
 * to the packed buffer and multiplied while on chip), then the top-k.
 * Results as ns_gather_head_rows followed by ns_sub_lm_head_logits_topk.
 */
NS_API ns_status ns_gather_sub_lm_head_topk(ns_handle *h, int32_t seq, const uint16_t *d_W_head,
                                            const uint16_t *d_hidden, int32_t n, int32_t k, float *d_logits,
                                            int32_t ld_logits, int32_t *d_topk_ids, float *d_topk_vals,
                                            ns_stream stream);

/*
 * The projection straight from W_head through I_t, with no packed copy: the
 * "naive indexed GEMM" of NanoSpec's ablation (evaluation, Table 5), kept
 * as a measured comparator.  The same tcgen05 kernel as
 * ns_gather_sub_lm_head_topk reads each W_head[I_t[j], :] in place and
 * stores nothing to the packed buffer.  Arguments and results as
 * ns_gather_sub_lm_head_topk (the packed buffer is left as it was).
 */
NS_API ns_status ns_sub_lm_head_indexed_topk(ns_handle *h, int32_t seq, const uint16_t *d_W_head,
                                             const uint16_t *d_hidden, int32_t n, int32_t k, float *d_logits,
                                             int32_t ld_logits, int32_t *d_topk_ids, float *d_topk_vals,
                                             ns_stream stream);

/*
 * CTAs of the copy kernels (ns_gather_head_rows, ns_gather_new_head_rows)
 * from now on; 0 restores the default (four per SM for the gather, two for
 * the slot-row copy).  A copy meant to run beside a backbone that fills the
 * GPU can take a few CTAs, which find room while the backbone's kernels hold
 * the rest.  Results do not depend on it.  NS_ERR_ARG for ctas < 0.
 */
NS_API ns_status ns_set_copy_ctas(ns_handle *h, int32_t ctas);

/*
 * ns_step with the step's inputs and outputs in host memory: the tree ids
 * (int32 [n_tree]), the verify row (fp32 [V], ignored when K_ver = 0) and
 * the hidden rows (bf16 [n x H]) in, the top-k ids and values (int32 / fp32
 * [n x k]) out to h_topk_ids / h_topk_vals, all on `stream` (logits in the
 * handle's scratch).  Page-locked buffers that the device can address (the
 * tree ids, the verify row, the outputs) are read and written by the step
 * kernel in place; other buffers, and always the hidden rows, go through
 * the handle's device staging by copies.  It returns once everything is
 * enqueued; the outputs are valid after the stream synchronises, and every
 * buffer must stay valid until then.  Pinned buffers also let the copies run
 * asynchronously.  d_W_head is device memory as in ns_step.  With trace
 * events set (ns_trace_events) the four events bracket the input copies,
 * the step and the output copies.  Arguments as in ns_step.
 */
NS_API ns_status ns_step_host(ns_handle *h, int32_t seq, const int32_t *h_tree_ids, int32_t n_tree,
                              const float *h_verify_row, const uint16_t *d_W_head, const uint16_t *h_hidden,
                              int32_t n, int32_t k, int32_t *h_topk_ids, float *h_topk_vals, ns_stream stream);

/*
 * Slot-stable packed buffer: the incremental reading of NanoSpec's
 * "Avoiding Sparse Computation via Asynchronous Gathering" (only the weights
 * of newly active tokens are gathered into the pre-allocated contiguous
 * buffer).  Each sequence has a second buffer of W_max row slots, separate
 * from the packed buffer above, and a table of the id each slot holds.
 *
 * ns_gather_new_head_rows updates the table to the current I_t (the one the
 * last ns_build_active_vocab / ns_state_update / ns_step produced) and copies
 * only the rows of the ids it places: every slot whose id left I_t is freed;
 * then the ids of I_t that hold no slot take the free slots in ascending id
 * order, lowest slot first (the pages fix no rule; this is the one used).
 * An id keeps its slot while it stays active.  ns_stream_init empties the
 * table, so the first update after it lays I_1 out ascending (as the full
 * repack does) and copies |I_1| rows; later updates copy |I_t \ I_{t-1}|.
 * Meant for a copy stream like ns_gather_head_rows: `done` (nullable) is
 * recorded on copy_stream after the copy.  d_W_head: bf16 [V x H].
 */
NS_API ns_status ns_gather_new_head_rows(ns_handle *h, int32_t seq, const uint16_t *d_W_head,
                                         ns_stream copy_stream, ns_event done);

/*
 * Projection and top-k over the slot buffer (tcgen05):
 *   logits[r, s] = sum_h hidden[r, h] * slot_row[s, h]  for s < high-water mark
 * (one past the highest occupied slot; columns of free slots below it hold
 * unspecified values and are never ranked), then per row the k largest logits
 * of occupied slots mapped to the ids they hold, ties to the smaller id.  The
 * ids and values equal those of ns_sub_lm_head_logits_topk on the same I_t;
 * only the logits' column order differs (by slot instead of by position in
 * I_t).  Arguments as ns_sub_lm_head_logits_topk (ld_logits >= W_max).
 */
NS_API ns_status ns_slot_lm_head_logits_topk(ns_handle *h, int32_t seq, const uint16_t *d_hidden, int32_t n,
                                             int32_t k, float *d_logits, int32_t ld_logits, int32_t *d_topk_ids,
                                             float *d_topk_vals, ns_stream stream);

/*
 * One decode step on the slot buffer, with the results of
 * ns_state_update, ns_gather_new_head_rows and ns_slot_lm_head_logits_topk
 * made in order on `stream` (the slot table, the slot rows, the copied-row
 * list and I_t included).  Arguments as ns_step; the logits are indexed by
 * slot, and columns of free slots below the high-water mark hold NaN.
 * When the slot table matches the window (the last call that changed this
 * sequence's window was a slot update: ns_gather_new_head_rows or
 * ns_step_slots) and the device holds the grid, it is ONE cooperative
 * launch (ns_step_slots_fused returns 1): the tiles of the occupied slots
 * are projected from the slot buffer while the window is updated, the ids
 * that enter take their slots and are projected by the draft item and the
 * verify products, and only their rows are copied.  Otherwise (after
 * ns_stream_init, ns_stream_append, ns_state_update, ns_step, ns_step_host
 * or a batched step) it is the three calls in order.
 */
NS_API ns_status ns_step_slots(ns_handle *h, int32_t seq, const int32_t *d_tree_ids, int32_t n_tree,
                               const float *d_verify_logits, int32_t n_verify, int32_t verify_row,
                               const uint16_t *d_W_head, const uint16_t *d_hidden, int32_t n, int32_t k,
                               float *d_logits, int32_t ld_logits, int32_t *d_topk_ids, float *d_topk_vals,
                               ns_stream stream);

/*
 * 1 when the next ns_step_slots on `seq` runs as one launch (the calls
 * enqueued so far leave the slot table matching the window, and the device
 * holds the grid), else 0 (also for a NULL handle or a bad seq).  Host
 * bookkeeping only; no device work.
 */
NS_API int32_t ns_step_slots_fused(const ns_handle *h, int32_t seq);

/*
 * Per-kernel event trace (MicroSpec §4 profiles per-step latency with CUDA
 * event recording).  While set, ns_step records, on its stream,
 *   events[0] before its first kernel,
 *   events[1] after the state update (append + active vocabulary),
 *   events[2] and events[3] after the fused gather + projection + top-k.
 * Inside stream capture they become external event nodes.  events must stay
 * valid while set; n_events must be 4, or 0 with events == NULL to switch
 * tracing off.  The events are borrowed cudaEvent_t.
 */
NS_API ns_status ns_trace_events(ns_handle *h, ns_event *events, int32_t n_events);

/*
 * Dense head on a fixed row range: logits over rows [0, rows) of W_head
 * (rows = V is the full-vocabulary LM head of Eq. 1; rows = 32768 a static
 * frequency-ranked sub-head) and per-row top-k with ids = row numbers.
 * Three launches: the projection on the tensor cores (whole 128-row tiles
 * of W_head by TMA, one persistent CTA per SM), then the top-k of 4096-column
 * slices of every row and their merge.  Uses the handle's dense scratch
 * (sized for V rows); the handle's V and H bound `rows` and fix H.
 * Arguments as in ns_sub_lm_head_logits_topk; ld_logits >= rows when
 * d_logits is not NULL.
 */
NS_API ns_status ns_dense_lm_head_topk(ns_handle *h, const uint16_t *d_W_head, int32_t rows,
                                const uint16_t *d_hidden, int32_t n, int32_t k, float *d_logits,
                                int32_t ld_logits, int32_t *d_topk_ids, float *d_topk_vals,
                                ns_stream stream);

/*
 * Dense head without any allocation (the paper has no counterpart: this is a
 * service for callers that cannot allocate device memory — code that lives
 * inside another framework's memory pool or a fixed memory budget, or a
 * plugin that is only handed pointers — and therefore cannot hold a handle,
 * because ns_create allocates).
 * Same arguments and results as ns_dense_lm_head_topk, with H given directly
 * instead of through a handle: logits over rows [0, rows) of W_head (bf16
 * [rows x H], 64 <= H <= 8192, H % 64 == 0) and per-row top-k with ids = row
 * numbers.  It calls no cudaMalloc/cudaFree and no allocating library
 * routine.  Its scratch is a fixed array of 6,291,456 bytes (6 MiB) inside
 * the library image, reserved on every GPU that loads the library until the
 * process exits.  It runs the same kernels as ns_dense_lm_head_topk, so the
 * logits and top-k are the handle's, bit for bit.  rows <= 2^19.  A bounded
 * wait that runs out is recorded in a word of the library image that no call
 * reads back.  `stream` must belong to the current device (NS_ERR_ARG
 * otherwise).  When d_logits is NULL the logits are kept in that scratch, which
 * holds at most NS_NOALLOC_MAX_LOGITS values: n * rows above that returns
 * NS_ERR_ARG (pass d_logits for larger heads, e.g. the full vocabulary).
 * The first call on each device looks up the scratch's device address and
 * prepares the kernels for that device; make that first call before any
 * stream capture.  Every call uses the same scratch and leaves its contents
 * behind: calls that may overlap on the GPU (different streams without an
 * ordering between them) race and must not be issued.
 */
#define NS_NOALLOC_MAX_LOGITS (1 << 20)
NS_API ns_status ns_dense_lm_head_topk_noalloc(const uint16_t *d_W_head, int32_t rows, int32_t H,
                                               const uint16_t *d_hidden, int32_t n, int32_t k, float *d_logits,
                                               int32_t ld_logits, int32_t *d_topk_ids, float *d_topk_vals,
                                               ns_stream stream);

/*
 * Device pointers into a sequence's state (owned by the handle; valid until
 * ns_destroy).  Any out-pointer may be NULL.
 *   ids     int32 [W_max]  I_t ascending (first *count entries valid)
 *   count   int32 [1]      |I_t|
 *   bitmap  uint32 [ceil(V/32)]  bit (i % 32) of word i / 32 set iff i in window
 *   packed  bf16 [W_max x H]     rows j < |I_t| valid after a gather
 */
NS_API ns_status ns_get_active(ns_handle *h, int32_t seq, const int32_t **ids, const int32_t **count,
                        const uint32_t **bitmap, const uint16_t **packed);

/*
 * Device pointers to the raw stream state (for inspection and tests):
 *   ring    int32 [W_max]  stream entry at position p lives at ring[p % W_max]
 *   length  int64 [1]      total number of entries ever appended (|S|)
 *   counts  uint32 [V]     occurrences of each id among the last W_max entries
 */
NS_API ns_status ns_get_state(ns_handle *h, int32_t seq, const int32_t **ring, const int64_t **length,
                       const uint32_t **counts);

/*
 * Checkpoint and resume of one sequence's stream state (not on the pages:
 * the state is the last W_max stream entries and |S|, everything else
 * follows from them).  The checkpoint is a 32-byte header (magic "NSST",
 * version 1, V, W_max, |S| as int64, n = min(|S|, W_max), 4 bytes reserved;
 * little-endian) followed by the window's n entries (int32), oldest first.
 *
 * ns_state_export_bytes: the largest checkpoint of this handle (header +
 * 4 * W_max bytes); 0 for NULL.
 *
 * ns_state_export writes the checkpoint of `seq` to host_buf (buf_bytes
 * long; NS_ERR_ARG when too short) and its size to *written; with host_buf
 * NULL it only writes the size.  It synchronises `stream` (the state is
 * read after the work queued on it).  NS_ERR_STATE before ns_stream_init.
 *
 * ns_state_import makes `seq` continue from a checkpoint: as ns_stream_init
 * it resets the sequence, then restores the ring and |S|, recounts the
 * window (counts, bitmap) and builds I_t, on `stream`.  The packed buffer is
 * not restored (the next ns_step or ns_gather_head_rows fills it) and the
 * slot table starts empty.  The host buffer is read before the call returns
 * (the call waits for the work queued on `stream` before its copy).
 * NS_ERR_ARG for a checkpoint of another V or W_max, a wrong magic, version
 * or size, or an id outside [0, V).
 */
NS_API int64_t ns_state_export_bytes(const ns_handle *h);
NS_API ns_status ns_state_export(ns_handle *h, int32_t seq, void *host_buf, int64_t buf_bytes, int64_t *written,
                                 ns_stream stream);
NS_API ns_status ns_state_import(ns_handle *h, int32_t seq, const void *host_buf, int64_t bytes, ns_stream stream);

/*
 * Device pointers to a sequence's slot buffer (owned by the handle).  Any
 * out-pointer may be NULL.
 *   slot_id    int32 [W_max]  id held by each slot, -1 = free
 *   meta       int32 [2]      high-water mark; rows copied by the last update
 *   new_slots  int32 [W_max]  slots the last update filled (first meta[1] valid),
 *   new_ids    int32 [W_max]  and the ids placed there, in ascending id order
 *   rows       bf16 [W_max x H]  slot s holds W_head[slot_id[s], :] when occupied
 */
NS_API ns_status ns_get_slots(ns_handle *h, int32_t seq, const int32_t **slot_id, const int32_t **meta,
                              const int32_t **new_slots, const int32_t **new_ids, const uint16_t **rows);

/* Synchronises the device, returns the sticky NS_FLAG_* mask, and clears it
 * when `clear` is non-zero. */
NS_API ns_status ns_get_error(ns_handle *h, uint32_t *flags, int32_t clear);

#ifdef __cplusplus
}
#endif

#endif /* NANOSPEC_H */
