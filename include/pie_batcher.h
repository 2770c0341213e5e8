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

/* Calls waiting in queues and calls in flight. */
int pie_batcher_counts(const pie_batcher_t* b, int64_t* queued, int64_t* in_flight);

#ifdef __cplusplus
}
#endif

#endif /* PIE_BATCHER_H_ */
