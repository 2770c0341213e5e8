/*
 * pie_fwd.h -- C ABI of the GB300 (sm_103a) ForwardPass hot path.
 *
 * One Pie ForwardPass carries many lanes in one launch ("The forward pass",
 * section Lanes): every lane has its own rows, concatenated and delimited by
 * a row offset array, and its own working set of KV pages.  For one
 * attention layer the pass
 *   1. rotates each row's q and k at the row's explicit position ID and
 *      writes the row's K/V into its slot of the lane's working set
 *      (section State geometry: positions, slots);
 *   2. runs grouped-query attention of every row over the lane's first
 *      kv_len slots, restricted by the row's slot mask when one is given
 *      (sections State geometry: kv_len; Attention masks);
 *   3. returns outputs for the readout rows, by default the last row of each
 *      lane (section Readouts);
 *   4. freezes each lane's `fold` newly written slots: none, all, a count,
 *      or a count that device code wrote into a channel (section State
 *      geometry, speculative decoding paragraph).
 * The four steps are the four calls pie_fwd_plan, pie_fwd_append_kv,
 * pie_fwd_attend and pie_fwd_fold, issued in that order on one stream
 * (section Pipelines and frames: passes on one pipeline run in submission
 * order).
 *
 * Conventions
 *   - Every device pointer is owned by the caller and must stay valid until
 *     the work queued on `stream` that uses it has finished.  `stream` is a
 *     cudaStream_t passed as void* (NULL = the legacy default stream).
 *   - Element types: PIE_F32 (float) or PIE_BF16 (bfloat16 stored as 16-bit
 *     words).  Arithmetic is fp32 on the GPU in both cases.
 *   - K/V pools are laid out [num_pool_pages][num_kv_heads][page_size]
 *     [head_dim], elements of the pass dtype.  Slot s of lane l lives in
 *     page page_ids[page_indptr[l] + s / page_size] at offset s % page_size.
 *   - Per-row tensors: q, q_rot [num_rows][num_q_heads][head_dim];
 *     k, v [num_rows][num_kv_heads][head_dim]; contiguous.
 *   - Mask words: slot s is visible to row r iff bit (s & 31) of
 *     mask_words[mask_word_indptr[r] + (s >> 5)] is set (LSB first).  A row
 *     needs at least ceil(kv_len / 32) words; bits at or past kv_len are
 *     ignored.  Without a mask a row sees slots s <= its own slot and
 *     s < kv_len (causal in slot space, which is the folding() geometry).
 *   - Every call returns PIE_OK (0) or a negative error code and queues no
 *     work on error.  pie_fwd_last_error() gives a message for the calling
 *     thread's last error.  No call synchronizes the host with the device.
 *   - Device-side findings are ORed into a caller-owned uint32 status word
 *     (PIE_STATUS_*); the caller reads it whenever convenient.
 *   - Kernels are launched with programmatic stream serialization: each may
 *     begin while the kernel queued before it on `stream` drains, and waits
 *     for that kernel (griddepcontrol.wait) before it reads what that kernel
 *     wrote.  The first kernel of every call waits at its start (the
 *     attention kernels first read only their plan's work items, uploaded by
 *     pie_fwd_plan before the pass's kernels), and no kernel lets the next
 *     one begin before its own wait has returned, so
 *     anything written by work queued earlier on `stream` is complete before
 *     any kernel of a call reads it: ordinary stream order is all a caller
 *     needs, and the caller's own kernels keep their usual semantics.
 */
#ifndef PIE_FWD_H_
#define PIE_FWD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- error codes -------------------------------------------------------- */
#define PIE_OK 0
#define PIE_EINVAL (-1)       /* malformed argument or metadata              */
#define PIE_ERANGE (-2)       /* a value outside its allowed range           */
#define PIE_ENOSPACE (-3)     /* workspace smaller than required             */
#define PIE_ECUDA (-4)        /* a CUDA runtime call failed                  */
#define PIE_EUNSUPPORTED (-5) /* dtype / head_dim / page_size not built      */

/* ---- element types ------------------------------------------------------ */
#define PIE_F32 0
#define PIE_BF16 1

/* ---- fold modes (StateGeometry.fold per lane) ---------------------------- */
#define PIE_FOLD_NONE 0    /* freeze nothing                                   */
#define PIE_FOLD_ALL 1     /* freeze every row written by this pass            */
#define PIE_FOLD_COUNT 2   /* freeze fold_count[l] rows (host literal)         */
#define PIE_FOLD_CHANNEL 3 /* freeze channel[l] rows, read on the device       */

/* ---- device status bits ---------------------------------------------------- */
#define PIE_STATUS_FROZEN_WRITE 1u /* a row's slot was frozen; its K/V write was skipped */
#define PIE_STATUS_FOLD_CLAMP 2u   /* a channel count outside [0, n] was clamped          */
#define PIE_STATUS_BOUNDS 4u       /* a device-supplied page id outside the pool, or a
                                      kv_len past the lane's pages, was skipped or cut
                                      (decode loop, no-allocation decode); outputs of the
                                      lanes concerned are invalid                         */
#define PIE_STATUS_FOLD_GAP 8u     /* a folding lane's first slot != its frozen length    */
#define PIE_STATUS_TIMEOUT 16u     /* a kernel's bounded wait expired; outputs invalid    */
#define PIE_STATUS_LOOP_FULL 64u     /* decode loop: a lane had no slot left for a token   */
#define PIE_STATUS_NOALLOC_TRUNC 32u /* no-allocation decode: a kv_len above max_kv_len was
                                        cut to max_kv_len                                   */

/* Static description of the attention layer. */
typedef struct pie_fwd_desc {
  int32_t num_q_heads;  /* Hq; a multiple of num_kv_heads                     */
  int32_t num_kv_heads; /* Hkv; q head h reads kv head h / (Hq / Hkv)          */
  int32_t head_dim;     /* d: 64 or 128                                        */
  int32_t page_size;    /* P: 8, 16 or 32 slots per KV page                     */
  int32_t dtype;        /* PIE_F32 or PIE_BF16                                  */
  float rope_base;      /* RoPE base (e.g. 10000); rotate-half pairing i, i+d/2 */
  float sm_scale;       /* softmax scale; 0 means 1 / sqrt(head_dim)            */
} pie_fwd_desc;

/* Per-pass metadata.  All arrays are HOST memory, read only during
 * pie_fwd_workspace_bytes / pie_fwd_plan and not retained. */
typedef struct pie_fwd_meta {
  int32_t num_lanes; /* L >= 0                                                 */
  int32_t num_rows;  /* N >= 0                                                 */
  const int32_t* row_indptr;  /* [L+1]: rows of lane l are [row_indptr[l], row_indptr[l+1]) */
  const int32_t* positions;   /* [N]: RoPE position ID of each row (>= 0)            */
  const int32_t* slots;       /* [N]: working-set slot each row writes               */
  const int32_t* kv_len;      /* [L]: slots the lane reads, <= its page capacity     */
  const int32_t* page_indptr; /* [L+1]: the lane's pages are page_ids[page_indptr[l]..] */
  const int32_t* page_ids;    /* physical page ids in [0, num_pool_pages)            */
  int32_t num_pool_pages;
  const int32_t* fold_mode;   /* [L]: PIE_FOLD_*                                     */
  const int32_t* fold_count;  /* [L]: used by PIE_FOLD_COUNT; may be NULL otherwise  */
  const int64_t* mask_word_indptr; /* [N+1] or NULL (default causal visibility)    */
  const int32_t* readout;     /* [R] row indices, or NULL: last row of every lane
                                 that has rows                                      */
  int32_t num_readout;        /* R when readout != NULL                              */
} pie_fwd_meta;

typedef struct pie_fwd_plan pie_fwd_plan_t;

/* Device workspace the plan needs for this pass (metadata, work lists and
 * split-softmax partials).  Host only; no CUDA call.
 * Errors: PIE_EINVAL / PIE_ERANGE / PIE_EUNSUPPORTED as pie_fwd_plan. */
int pie_fwd_workspace_bytes(const pie_fwd_desc* desc, const pie_fwd_meta* meta,
                            size_t* bytes);

/* Plan one pass (the "state" and "mask"/"readout" set-up of a ForwardPass).
 * Validates the metadata:
 *   PIE_EINVAL  - non-monotone or inconsistent indptr arrays, unknown fold
 *                 mode, two rows writing the same physical slot (the
 *                 hazard-freedom condition of the Pie review, Eq. (4)), or a
 *                 folding lane whose slots are not consecutive;
 *   PIE_ERANGE  - negative position, slot outside the lane's pages, kv_len
 *                 above the lane's capacity, page id outside the pool,
 *                 readout row out of range, fold_count outside [0, n], or a
 *                 row with fewer than ceil(kv_len/32) mask words;
 *   PIE_EUNSUPPORTED - head_dim / page_size / dtype not built;
 *   PIE_ENOSPACE - ws_bytes < pie_fwd_workspace_bytes().
 * Builds the work lists on the host and queues one host-to-device copy into
 * `dev_workspace` (256-byte aligned, caller-owned, must outlive the plan's
 * use) on `stream`.  The returned plan is immutable, owned by the library,
 * usable for any number of append/attend/fold calls on streams ordered after
 * `stream`, and released with pie_fwd_plan_destroy. */
int pie_fwd_plan(const pie_fwd_desc* desc, const pie_fwd_meta* meta, void* dev_workspace,
                 size_t ws_bytes, void* stream, pie_fwd_plan_t** out);

/* Number of readout rows R of a plan (the first dimension of out_readout). */
int32_t pie_fwd_plan_num_readout(const pie_fwd_plan_t* plan);

/* Step 1 (State geometry: positions, slots).  For every row r of lane l:
 *   q_rot[r,h]  = RoPE(q[r,h], positions[r])                 for all q heads
 *   K_pool[slot] = RoPE(k[r,g], positions[r]), V_pool[slot] = v[r,g]
 * RoPE pairs element i with i + d/2 at angle positions[r] * base^(-2i/d)
 * (fp32 angle).  A row whose slot is below frozen_len[l] is not written and
 * sets PIE_STATUS_FROZEN_WRITE; a lane with fold != NONE whose first slot is
 * not frozen_len[l] sets PIE_STATUS_FOLD_GAP.
 * q, k, v: device, read; q_rot: device [N,Hq,d], written; k_pool, v_pool:
 * device pools, written at the rows' slots only; frozen_len: device int32 [L];
 * status: device uint32 (may be NULL).  Errors: PIE_EINVAL on a NULL
 * required pointer, PIE_ECUDA on a failed launch. */
int pie_fwd_append_kv(const pie_fwd_plan_t* plan, const void* q, const void* k, const void* v,
                      void* q_rot, void* k_pool, void* v_pool, const int32_t* frozen_len,
                      uint32_t* status, void* stream);

/* Step 2-3 (State geometry: kv_len; Attention masks; Readouts).  For every
 * row r of lane l and q head h (kv head g = h / (Hq/Hkv)), over the visible
 * slots V(r) of [0, kv_len[l]):
 *   z_s = sm_scale * <q_rot[r,h], K[s,g]>,  o = sum_s softmax(z)_s V[s,g],
 *   lse = log(sum_s exp(z_s)).
 * An empty V(r) gives o = 0 and lse = -inf.
 * mask_words: device uint32 words (required iff the plan has a mask).
 * out_readout: device [R,Hq,d] in the dtype (may be NULL if R == 0);
 * lse_readout: device float [R,Hq] or NULL; out_all: device [N,Hq,d] or
 * NULL (every row's output); lse_all: device float [N,Hq] or NULL.
 * The pools are only read.  Precondition: every slot below kv_len holds
 * finite K and V (masked-out slots included); slots at or past kv_len may
 * hold anything.  status: device uint32 or NULL (PIE_STATUS_TIMEOUT).
 * Calls on one plan share its workspace (the split partials, and the work
 * counter from which the split-KV kernel's persistent grid takes its items):
 * queue them one after another (one per layer, on one stream or ordered by
 * events), never concurrently. */
int pie_fwd_attend(const pie_fwd_plan_t* plan, const void* q_rot, const void* k_pool,
                   const void* v_pool, const uint32_t* mask_words, void* out_readout,
                   float* lse_readout, void* out_all, float* lse_all, uint32_t* status,
                   void* stream);

/* The pass's attention mask, once for every layer ("The forward pass",
 * Attention masks: the mask belongs to the ForwardPass, and every attention
 * layer of the pass applies it).  For bf16 lanes with head_dim 128 (decode
 * rows and prefill alike), attention walks, per row block, a compacted list of
 * the slots some row of the block sees (and each row's mask re-expressed over
 * that list), built
 * from the mask words and the page table -- data of the pass, not of the
 * layer.  pie_fwd_set_mask builds those lists on `stream` into the plan's
 * workspace and records `mask_words`; every later pie_fwd_attend call on this
 * plan given the same mask_words pointer reuses them instead of building them
 * again (so an L-layer model builds them once, not L times).  The words must
 * not change while the plan uses them; an attend call given another pointer
 * builds the lists itself, as it does when set_mask was never called.
 * mask_words: device uint32 words, as for pie_fwd_attend.  Not thread-safe
 * with other calls on the same plan.  Errors: PIE_EINVAL (NULL plan or
 * words, a plan without a mask), PIE_ECUDA (launch). */
int pie_fwd_set_mask(pie_fwd_plan_t* plan, const uint32_t* mask_words, void* stream);

/* Step 4 (State geometry: fold).  frozen_len[l] += k_l with k_l = 0 (NONE),
 * n_l (ALL), fold_count[l] (COUNT) or clamp(channel[l], 0, n_l) (CHANNEL;
 * PIE_STATUS_FOLD_CLAMP when clamped).  channel: device int32 [L], written
 * earlier on `stream` (required iff a lane uses PIE_FOLD_CHANNEL). */
int pie_fwd_fold(const pie_fwd_plan_t* plan, int32_t* frozen_len, const int32_t* channel,
                 uint32_t* status, void* stream);

/* Releases a plan.  Waits for the plan's own host-to-device copy if it is
 * still in flight; never waits for kernels. */
void pie_fwd_plan_destroy(pie_fwd_plan_t* plan);

/* One whole ForwardPass (steps 1-4 of "The forward pass") in one call, on
 * `stream`: pie_fwd_plan into dev_workspace, pie_fwd_append_kv,
 * pie_fwd_set_mask when the pass has a mask, pie_fwd_attend, pie_fwd_fold,
 * then pie_fwd_plan_destroy (the plan's pinned staging is reused only after
 * its upload completed).  Every argument means what it means in those calls;
 * mask_words and channel are NULL when the pass has neither.  The workspace
 * is busy until the pass's kernels have finished: a caller that plans the
 * next pass on another stream first waits for an event recorded after this
 * call.  Errors: those of the calls, from the first that fails (nothing later
 * is launched). */
int pie_fwd_forward(const pie_fwd_desc* desc, const pie_fwd_meta* meta, void* dev_workspace,
                    size_t ws_bytes, const void* q, const void* k, const void* v, void* q_rot,
                    void* k_pool, void* v_pool, int32_t* frozen_len, const uint32_t* mask_words,
                    void* out_readout, float* lse_readout, void* out_all, float* lse_all,
                    const int32_t* channel, uint32_t* status, void* stream);

/* Message for the calling thread's most recent error ("" if none). */
const char* pie_fwd_last_error(void);

/* Readout distribution epilogue (the review "Pie: Who Should Control the
 * LLM Generation Loop?", section 7, Eq. (6)-(7): the serving system returns
 * the K most probable tokens of the next-token distribution, K = 256 by
 * default, and the mass Z they keep; 1 - Z is the total-variation distance
 * of Eq. (7) when a client renormalises them).
 *   logits : device, `rows` rows of `vocab` logits of `dtype` (PIE_F32 or
 *            PIE_BF16), row r at logits + r * ld elements; rows start on
 *            16-byte boundaries (logits 16-byte aligned, ld * element size a
 *            multiple of 16); finite values or -inf.
 *   ids    : device int32 [rows][k]: for each row the k tokens of largest
 *            p = softmax(logits row) (temperature 1), largest first, equal
 *            logits by smaller token id first.
 *   probs  : device fp32 [rows][k]: p of those tokens (not renormalised).
 *   z      : device fp32 [rows] or NULL: Z = the sum of the row's probs.
 *   lse    : device fp32 [rows] or NULL: log(sum_v exp(logit_v)).
 *   workspace : device, 256-byte aligned, at least
 *            pie_fwd_readout_topk_workspace_bytes() bytes, caller-owned.
 * Supported: 1 <= k <= 256, k <= vocab <= 262,144 (PIE_EUNSUPPORTED
 * beyond); PIE_EINVAL for a bad dtype, NULL logits/ids/probs, ld < vocab or
 * misaligned rows; PIE_ENOSPACE for a short workspace.  Four kernels on
 * `stream` (a sampled bound, one pass over the logits, an exact fallback for
 * rows the bound does not serve, the merge); no host synchronization. */
int pie_fwd_readout_topk_workspace_bytes(int32_t dtype, int32_t rows, int32_t vocab, int32_t k,
                                         size_t* bytes);
int pie_fwd_readout_topk(const void* logits, int32_t dtype, int32_t rows, int32_t vocab,
                         int64_t ld, int32_t k, int32_t* ids, float* probs, float* z,
                         float* lse, void* workspace, size_t ws_bytes, void* stream);

/* Decode loop that runs ahead of the host ("The forward pass", Pipelines and
 * frames: run_ahead keeps a repeating decode pass in flight on the GPU).
 * Runs `steps` single-row passes per lane on `stream`; step t of lane l is
 * the folding() geometry of one new token (State geometry): position = slot
 * = frozen_len[l], kv_len = frozen_len[l] + 1, fold all (frozen_len[l] += 1).
 * The geometry and the work items are derived on the device from
 * frozen_len, so the call builds no host plan per token, allocates nothing,
 * never synchronizes the host and may be captured in a CUDA graph.
 *   page_indptr [L+1], page_ids: device, the lanes' page lists (as in
 *            pie_fwd_meta); each lane's capacity is its pages x page_size.
 *   num_pool_pages: host, pages per pool; the kernels check every page id
 *            they read against it (an id outside [0, num_pool_pages) is
 *            neither written nor read and sets PIE_STATUS_BOUNDS).
 *   max_pages_per_lane: host, a bound on every lane's page count (sizes the
 *            work-item grid and the workspace).
 *   frozen_len [L]: device int32, read and advanced on the device.
 *   q [steps][L][Hq][d], k, v [steps][L][Hkv][d]: device, per-step inputs
 *            of the pass dtype; q_rot [L][Hq][d]: device scratch (the last
 *            step's rotated queries on return).
 *   out [steps][L][Hq][d] (pass dtype), lse [steps][L][Hq] (fp32, or NULL):
 *            each step's attention output of every lane.
 *   channel [steps][L]: device int32, or NULL (every step folds its token).
 *            Step t of lane l freezes clamp(channel[t][l], 0, 1) slots (State
 *            geometry, speculative-decoding paragraph: the accepted count comes
 *            from a device channel; out-of-range counts are clamped and set
 *            PIE_STATUS_FOLD_CLAMP).  A lane that freezes 0 keeps its frozen
 *            length, so its next step writes the same slot at the same
 *            position and the rejected token is overwritten before it is read.
 *            channel[t] must be written on `stream` before step t's fold.
 *   workspace: device, 256-byte aligned, at least
 *            pie_fwd_decode_loop_workspace_bytes(); status: device uint32 or
 *            NULL.
 * A lane with no slot left (frozen_len >= its capacity) writes nothing, gets
 * o = 0 and lse = -inf, does not advance, and sets PIE_STATUS_LOOP_FULL.
 * Errors as pie_fwd_plan / pie_fwd_append_kv for shapes and pointers. */
int pie_fwd_decode_loop_workspace_bytes(const pie_fwd_desc* desc, int32_t num_lanes,
                                        int32_t max_pages_per_lane, size_t* bytes);
int pie_fwd_decode_loop(const pie_fwd_desc* desc, int32_t num_lanes, int32_t steps,
                        const int32_t* page_indptr, const int32_t* page_ids,
                        int32_t num_pool_pages, int32_t max_pages_per_lane,
                        int32_t* frozen_len, const void* q,
                        const void* k, const void* v, void* q_rot, void* k_pool, void* v_pool,
                        void* out, float* lse, const int32_t* channel, void* workspace,
                        size_t ws_bytes, uint32_t* status, void* stream);

/* Per-lane adapters at a projection site ("The forward pass", section
 * Adapters: an adapter is a function of a projection's input x and base
 * output y, LoRA adds b (a x), IA3 scales y, and requests in one batch may
 * use different adapters).  Every row of lane l takes adapter
 * a = adapter_of_lane[l] (-1: none) and becomes
 *     y' = (y + scale[a] * B_a (A_a x)) * s_a      (elementwise in s_a)
 * with A_a = lora_a[a] [rank][d_in], B_a = lora_b[a] [d_out][rank] and
 * s_a = ia3[a] [d_out] (all ones when ia3 is NULL).  y is updated in place;
 * rows of lanes without an adapter are not touched.  Products and sums are
 * fp32 (A_a x on the tensor cores from bf16 operands), y' is rounded to bf16
 * once.
 *
 * A plan cuts the lanes' rows into tiles of up to 128 consecutive rows of one
 * lane; it depends only on the lanes, so one plan serves every site and layer
 * of a pass (q, k, v, o, gate_up, down), each with its own weights and dims.
 *   row_indptr [L+1], adapter_of_lane [L]: HOST arrays, read during the call
 *            and not retained; rows of lane l are [row_indptr[l], row_indptr[l+1]).
 *   max_rank: the largest rank any apply of this plan will use.
 *   dev_workspace: device, 256-byte aligned, at least
 *            pie_fwd_adapter_workspace_bytes(); holds the tiles (one
 *            host-to-device copy queued on `stream`) and the fp32 partial
 *            sums of A_a x.  Applies of one plan share that scratch: issue them
 *            on one stream (or otherwise ordered).
 * Errors: PIE_EINVAL (NULL arrays, row_indptr[0] != 0 or not monotone),
 * PIE_ERANGE (adapter id outside [-1, num_adapters)), PIE_EUNSUPPORTED
 * (max_rank not in {0, 8, 16, 32, 64}), PIE_ENOSPACE (short workspace). */
typedef struct pie_fwd_adapter_plan pie_fwd_adapter_plan_t;
int pie_fwd_adapter_workspace_bytes(int32_t num_lanes, const int32_t* row_indptr,
                                    int32_t max_rank, size_t* bytes);
int pie_fwd_adapter_plan(int32_t num_lanes, const int32_t* row_indptr,
                         const int32_t* adapter_of_lane, int32_t num_adapters, int32_t max_rank,
                         void* dev_workspace, size_t ws_bytes, void* stream,
                         pie_fwd_adapter_plan_t** out);
/* Number of tiles of a plan (rows of lanes with an adapter, 128 per tile). */
int32_t pie_fwd_adapter_plan_num_tiles(const pie_fwd_adapter_plan_t* plan);
/* Number of adapter groups when every adapter in use serves at most 16 rows
 * (a decode-shaped plan): each apply with rank > 0 then runs one kernel, a
 * cluster of 8 CTAs per group; 0 when the plan applies by tiles (two kernels,
 * shrink and expand).  -1 for a NULL plan. */
int32_t pie_fwd_adapter_plan_num_groups(const pie_fwd_adapter_plan_t* plan);
/* Apply the adapters at one site.
 *   x: device bf16 [num_rows][d_in]; y: device bf16 [num_rows][d_out], both
 *            contiguous and 16-byte aligned.
 *   lora_a: device bf16 [num_adapters][rank][d_in]; lora_b: device bf16
 *            [num_adapters][d_out][rank]; scale: device fp32 [num_adapters];
 *            ia3: device bf16 [num_adapters][d_out] or NULL.  With rank 0 only
 *            the IA3 scaling runs (x, lora_a, lora_b, scale may be NULL).
 *   status: device uint32 or NULL (PIE_STATUS_TIMEOUT).
 * Supported: dtype PIE_BF16, rank in {0, 8, 16, 32, 64} and <= max_rank,
 * d_in a multiple of 64, d_out a multiple of 256 (PIE_EUNSUPPORTED / ERANGE
 * otherwise); PIE_EINVAL for NULL or misaligned required pointers.  Up to two
 * kernels on `stream` (one for a grouped plan, see
 * pie_fwd_adapter_plan_num_groups); no host synchronization. */
int pie_fwd_adapter_apply(const pie_fwd_adapter_plan_t* plan, int32_t dtype, int32_t d_in,
                          int32_t d_out, int32_t rank, const void* x, void* y, const void* lora_a,
                          const void* lora_b, const float* scale, const void* ia3,
                          uint32_t* status, void* stream);
/* Release a plan (its staging memory is reused once its upload completed). */
void pie_fwd_adapter_plan_destroy(pie_fwd_adapter_plan_t* plan);

/* Measurement hook (no counterpart on the Pie pages: it only lets a caller
 * time the attention kernels apart from the rest of a call).  After
 * pie_fwd_set_timing_events(start, stop) with two timing-enabled cudaEvent_t
 * handles, every pie_fwd_attend call made by the calling thread records
 * `start` on its stream right before its attention kernels (split-KV and/or
 * tensor-core) and `stop` right after them; the mask pre-pass and the
 * combine step fall outside.  Every pie_fwd_readout_topk call records them
 * around its pass over the logits (the stream kernel); the sample, slice and
 * merge steps fall outside.  The events stay caller-owned; (NULL, NULL)
 * turns the hook off.  Returns PIE_EINVAL when exactly one is NULL. */
int pie_fwd_set_timing_events(void* start_event, void* stop_event);

/* Test hook (the Pie pages have no counterpart: it exists so that tests can
 * run the bounded-wait failure path without faulting or hanging a GPU).  After
 * pie_fwd_test_wait_expiry(stage, wait_us) with stage >= 0, every split-KV
 * attention kernel that the calling thread launches (pie_fwd_attend, the
 * decode loop, the no-allocation decode) has its producer warp stop before
 * stage `stage` of a work item -- so no copy of that stage, or of any later
 * one, is ever in flight (a CTA that walks several items issues nothing for
 * its later items) -- and gives each of its waits `wait_us` microseconds: the
 * compute warps' wait for that stage expires, the kernel sets
 * PIE_STATUS_TIMEOUT, writes whatever partial state it has and returns.
 * Items with fewer stages that a CTA walks first are not affected.  (-1, 0)
 * turns the hook off.
 * Errors: PIE_EINVAL for stage < -1, or stage >= 0 with wait_us == 0. */
int pie_fwd_test_wait_expiry(int32_t stage, uint32_t wait_us);

/* ABI version of this header (major * 100 + minor). */
int pie_fwd_abi_version(void);

/* Decode attention that allocates nothing.  The Pie pages have no
 * counterpart for this call: it is a deployment variant of the split-KV
 * attention and combine steps of pie_fwd_attend for callers that cannot
 * allocate device memory when they launch attention (for example code
 * running under a foreign memory manager with a fixed device budget, or a
 * host path that must not take the allocator's locks), and so cannot provide
 * the plan workspace.
 *
 * One query row per lane: row l attends, with default visibility, over slots
 * [0, min(kv_len[l], slots[l] + 1)) of lane l's working set, exactly as
 * pie_fwd_attend does for a plan whose lanes have one row each.
 *   slots, kv_len: device int32 [num_lanes]; page_indptr: device int32
 *   [num_lanes + 1]; page_ids: device int32 (pool layout as above);
 *   num_pool_pages: pages per pool.  These arrays are device data, so they
 *   are checked on the device: a lane's extent is cut to the slots its pages
 *   hold, and a page id outside [0, num_pool_pages) is not read; either sets
 *   PIE_STATUS_BOUNDS (that lane's output is then invalid);
 *   q_rot: device [num_lanes][Hq][d] (e.g. from pie_fwd_append_kv);
 *   k_pool, v_pool: device pools, read only;
 *   out: device [num_lanes][Hq][d] in the dtype; lse: device float
 *   [num_lanes][Hq] or NULL; status: device uint32 or NULL.
 *   max_kv_len: host upper bound of kv_len (sizes the launch); larger device
 *   values are cut to it and set PIE_STATUS_NOALLOC_TRUNC.
 * Scratch lives in one static __device__ array of 16 MiB that every GPU
 * loading the library holds until exit; a call needing more
 * (num_lanes * num_kv_heads * ceil(max_kv_len / 512) * partial states)
 * returns PIE_ERANGE.  The first call on each device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current, so make
 * it before any stream capture.  Every call reuses the same array: calls
 * whose executions overlap on the GPU race; issue them on one stream.
 * Calls no allocator (no cudaMalloc, cudaFree or allocating library).
 * Errors: PIE_EINVAL (NULL pointer, bad head counts, negative size),
 * PIE_EUNSUPPORTED (shape), PIE_ERANGE (scratch), PIE_ECUDA (launch). */
int pie_fwd_decode_attend_noalloc(const pie_fwd_desc* desc, int32_t num_lanes,
                                  int32_t max_kv_len, const int32_t* slots,
                                  const int32_t* kv_len, const int32_t* page_indptr,
                                  const int32_t* page_ids, int32_t num_pool_pages,
                                  const void* q_rot,
                                  const void* k_pool, const void* v_pool, void* out,
                                  float* lse, uint32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PIE_FWD_H_ */
