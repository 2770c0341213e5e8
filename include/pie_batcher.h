/*
 * pie_batcher.h -- work-conserving dispatch of GPU-bound API calls.
 *
 * The host step before pie_fwd_plan: calls wait in command queues and, each
 * time the GPU goes idle, one batch is formed and dispatched (the Pie review,
 * section 5 "Batching API calls while preserving meaning": Algorithm 2, Eq. (4),
 * horizontal batching across queues and vertical batching within a queue).
 *   - A queue contributes only through its oldest pending call, once every
 *     dependency of that call has completed (queue order is kept).
 *   - For handler types that keep order inside a batch ("ordered", e.g. a
 *     forward pass, whose scatter runs before its attention), the following
 *     calls of the same queue and type join the head as a vertical group while
 *     each one's dependencies have completed or are earlier in the group.
 *   - Groups of one handler type are taken in queue-priority order (higher
 *     first, then the group holding the older call); a group joins only if
 *     Eq. (4) holds between its read/write sets and those of every group
 *     already taken: W(a) & (R(b) | W(b)) and W(b) & (R(a) | W(a)) are empty.
 *   - The ordered calls are cut at the first call that would exceed max_calls
 *     or max_rows; a batch always keeps its first call.
 *   - Between handler types, the batch holding the oldest pending call wins.
 *   - Consecutive calls of one group with the same working-set key (>= 0)
 *     form one lane of the pass (a prefix forward and its continuation); every
 *     other call is a lane of its own.
 * Call ids are assigned in arrival order from 0; they are the calls' age.
 *
 * Every function returns PIE_OK (0) or a negative PIE_E* code of pie_fwd.h
 * and changes nothing on error.  A batcher is not thread-safe: one control
 * thread owns it.  No CUDA call is made.  Ids are never reused: a completed
 * call keeps a record of about 100 bytes (its dependency and resource lists
 * are freed), so a long-lived control layer starts a new batcher when the
 * record count matters.
 */
#ifndef PIE_BATCHER_H_
#define PIE_BATCHER_H_

#include <stddef.h>
#include <stdint.h>

#include "pie_fwd.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pie_batcher pie_batcher_t;

/* ordered[h] != 0: handler type h forms vertical groups (0 <= h < num_handlers).
 * max_calls >= 1 and max_rows >= 1 are the backend's batch limits.
 * Errors: PIE_EINVAL (NULL out, num_handlers < 1, a limit < 1). */
int pie_batcher_create(int32_t num_handlers, const uint8_t* ordered, int32_t max_calls,
                       int64_t max_rows, pie_batcher_t** out);
void pie_batcher_destroy(pie_batcher_t* b);

/* A new command queue of the given priority (higher goes first inside a batch);
 * its id is written to *queue_id (0, 1, 2, ...). */
int pie_batcher_add_queue(pie_batcher_t* b, int32_t priority, int32_t* queue_id);

/* Enqueue a call (Algorithm 2's arrival step).  rows >= 1 counts against
 * max_rows; key >= 0 names its working set (-1: none); deps are ids of earlier
 * calls; reads / writes are resource ids in [0, 2^26) (e.g. KV page ids; the
 * batcher keeps a table indexed by resource id), any order, duplicates
 * allowed.  Arrays may be NULL when their count is 0.  The call's id goes to
 * *call_id.  Errors: PIE_EINVAL (unknown queue or handler, rows < 1, a
 * dependency that is not an earlier call, negative counts), PIE_ERANGE (a
 * resource id outside [0, 2^26)). */
int pie_batcher_submit(pie_batcher_t* b, int32_t queue, int32_t handler, int64_t rows,
                       int64_t key, const int64_t* deps, int32_t num_deps,
                       const int64_t* reads, int32_t num_reads, const int64_t* writes,
                       int32_t num_writes, int64_t* call_id);

/* Enqueue n calls at once, as n calls of pie_batcher_submit in order: call i
 * (0 <= i < n) takes queues[i], handlers[i], rows[i], keys[i] and the lists
 * deps[dep_indptr[i] .. dep_indptr[i+1]), reads[read_indptr[i] ..
 * read_indptr[i+1]), writes[write_indptr[i] .. write_indptr[i+1]) (offset
 * arrays of n + 1 entries from 0, never decreasing; a flat array may be NULL
 * when its offsets end at 0).  Call i gets id *first_id + i, so a dependency
 * may name a call earlier in the same submission.  Every call is checked
 * before any is enqueued: on error nothing changes.  Errors as
 * pie_batcher_submit, and PIE_EINVAL for NULL per-call arrays or bad offset
 * arrays. */
int pie_batcher_submit_many(pie_batcher_t* b, int32_t n, const int32_t* queues,
                            const int32_t* handlers, const int64_t* rows, const int64_t* keys,
                            const int64_t* dep_indptr, const int64_t* deps,
                            const int64_t* read_indptr, const int64_t* reads,
                            const int64_t* write_indptr, const int64_t* writes,
                            int64_t* first_id);

/* Form and dispatch one batch (Algorithm 2's GPU-idle step): its call ids in order go to
 * calls[0..n), the lane of each call to lanes[0..n) (0, 1, ...), its handler
 * type to *handler, n to *num_calls (0 and handler -1 when no call is
 * eligible).  The calls count as in flight until completed.  capacity is the
 * length of calls and lanes; Errors: PIE_ENOSPACE if capacity < max_calls. */
int pie_batcher_dispatch(pie_batcher_t* b, int64_t* calls, int32_t* lanes, int32_t capacity,
                         int32_t* num_calls, int32_t* handler);

/* Completion events (Algorithm 2's completion step): the calls have finished on the GPU, so calls
 * that depend on them become eligible.  Errors: PIE_EINVAL if a call is not in
 * flight (unknown, still queued or already completed); nothing is changed. */
int pie_batcher_complete(pie_batcher_t* b, const int64_t* calls, int32_t n);

/* ---- forward calls on registered working sets ------------------------------
 * A working set (a lane's KV state, Pie "The forward pass": State geometry) is
 * a list of pool pages in slot order: slot s lies in page pages[s / page_size].
 * The batcher keeps these lists so that the control loop hands it no per-page
 * data per call: a forward call's read set is the pages holding every slot up
 * to its last row's, its write set the pages holding its new slots (the sets
 * Eq. (4) compares), and a dispatched batch of forward calls becomes the
 * geometry of one pass without a host-side copy loop. */

/* Registers (or replaces) the page list of working set `key` (0 <= key <
 * 2^26; page ids in [0, 2^26)).  The list is copied.  Calls already queued
 * keep the read/write sets they were given.  Errors: PIE_EINVAL (NULL batcher,
 * negative count, NULL pages with a positive count), PIE_ERANGE (key or a page
 * id outside [0, 2^26)). */
int pie_batcher_set_pages(pie_batcher_t* b, int64_t key, const int32_t* pages, int32_t num_pages);

/* Enqueue n forward calls of handler type `handler`, as n calls of
 * pie_batcher_submit without dependencies: call i (ids *first_id + i) goes to
 * queues[i], names working set keys[i] (registered) and writes rows[i] >= 1
 * rows at slots [first_slot[i], first_slot[i] + rows[i]); it reads the pages
 * of slots [0, first_slot[i] + rows[i]) and writes the pages of its new slots.
 * Every call is checked before any is enqueued.  Errors: as
 * pie_batcher_submit; PIE_EINVAL for NULL arrays, page_size < 1 or a key with
 * no registered pages; PIE_ERANGE for slots past the working set's pages. */
int pie_batcher_submit_forward(pie_batcher_t* b, int32_t n, const int32_t* queues, int32_t handler,
                               const int64_t* keys, const int64_t* rows, const int64_t* first_slot,
                               int32_t page_size, int64_t* first_id);

/* The pass of a dispatched batch of forward calls (calls[0..n), lanes[0..n) as
 * pie_batcher_dispatch returned them), in pie_fwd_meta's layout: lane l holds
 * the calls numbered l, all on one working set k = lane_keys[l] (a working set
 * appears in one lane); its rows are its calls' rows concatenated in batch
 * order at slots frozen[k], frozen[k] + 1, ... (position = slot, so the
 * output arrays `positions` serve as slots too), kv_len[l] = frozen[k] + rows,
 * and its pages are the working set's registered pages.  first_row[i] is call
 * i's first row in the pass.  frozen[0..num_keys) is the caller's frozen length
 * per key.  Every pass folds all of its rows (PIE_FOLD_ALL).  Outputs:
 * row_indptr [L+1], positions [N], kv_len [L], page_indptr [L+1], page_ids
 * [pages], lane_keys [L] with L <= max_lanes, N <= max_rows, pages <=
 * max_pages; *num_lanes, *num_rows and *num_pages are set even when the
 * capacities are too small (then PIE_ENOSPACE and nothing else is written).
 * Errors: PIE_EINVAL (NULL arguments, an unknown call, a lane outside [0, n)
 * or holding no call, a lane spanning two working sets, a working set in two
 * lanes, a key with no registered pages or >= num_keys), PIE_ERANGE (negative
 * frozen length, a pass over 2^31 rows or pages), PIE_ENOSPACE.  No CUDA call;
 * the batcher is not changed. */
int pie_batcher_forward_pass(const pie_batcher_t* b, const int64_t* calls, const int32_t* lanes,
                             int32_t n, const int32_t* frozen, int64_t num_keys, int32_t max_lanes,
                             int64_t max_rows, int64_t max_pages, int32_t* row_indptr,
                             int32_t* positions, int32_t* kv_len, int32_t* page_indptr,
                             int32_t* page_ids, int64_t* lane_keys, int32_t* first_row,
                             int32_t* num_lanes, int32_t* num_rows, int64_t* num_pages);

/* pie_batcher_forward_pass and pie_fwd_plan (pie_fwd.h) in one call: the pass
 * of a dispatched forward batch is built in the batcher's own buffers and
 * planned against `desc`, `num_pool_pages`, the workspace and the stream as
 * pie_fwd_plan does (no fold count, mask or readout list: the default readout
 * of the last row of every lane).  Outputs: *plan, lane_keys [n] (the working
 * set of each lane), first_row [n], kv_len [n] (may be NULL), *num_lanes,
 * *num_rows.  Errors: those of both calls, PIE_EINVAL for n < 1; *plan is NULL
 * on error. */
int pie_batcher_plan_forward(pie_batcher_t* b, const int64_t* calls, const int32_t* lanes, int32_t n,
                             const int32_t* frozen, int64_t num_keys, const pie_fwd_desc* desc,
                             int32_t num_pool_pages, void* dev_workspace, size_t ws_bytes,
                             void* stream, pie_fwd_plan_t** plan, int64_t* lane_keys,
                             int32_t* first_row, int32_t* kv_len, int32_t* num_lanes,
                             int32_t* num_rows);

/* Calls waiting in queues and calls in flight. */
int pie_batcher_counts(const pie_batcher_t* b, int64_t* queued, int64_t* in_flight);

#ifdef __cplusplus
}
#endif

#endif /* PIE_BATCHER_H_ */
