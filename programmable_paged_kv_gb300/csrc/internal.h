// Internal structures shared by the host planner and the CUDA kernels of the
// ForwardPass hot path.  Not part of the public ABI (include/pie_fwd.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "pie_fwd.h"

namespace pie {

// Work item of the split-KV attention kernel: the queries of rows
// [row0, row0 + nrows) of `lane` that read kv head `kv_head` (nrows * G query
// vectors, padded to the kernel's NQ), over the slot chunk [kv_begin, kv_end).
// kv_begin is a multiple of kStageSlots.  Partial softmax state goes to
// partial slots part_base .. part_base + NQ - 1.  In masked passes `block` is
// the row block whose compacted visible-slot list the item walks (else -1);
// then kv_begin is the item's chunk and kv_end the chunks provisioned, and the
// chunks used come from the list's length (masked_chunks).
struct alignas(16) DecItem {
  int32_t lane, kv_head, row0, nrows;
  int32_t kv_begin, kv_end, part_base, block;
};

// The split-KV kernel keeps three CTAs per SM: a masked unit on it splits its
// list for two waves of three CTAs per SM (so that each CTA's start-up -- its
// item, the list length, the first copies -- partly runs under other CTAs'
// streaming; one wave, three or five measured slower), where a tensor-core
// unit splits for one wave of one.
constexpr int kDecListWaves = 6;
// The tensor-core split-KV kernel runs an item's start-up under the item
// before.  Plain passes: a persistent grid takes items from a counter (the
// decode batch 3.5 % faster than one item per CTA; fixed runs of two items
// lengthen its last wave and were 3.5 % slower).  List passes: fixed runs of
// two consecutive items per CTA (masked decode 3-5 % faster than one; the
// counter gave the same kernel times and slower calls).
constexpr int kDecListItemsPerCta = 2;

// How the combine step finds the partials of a row block (the rows one work
// item serves) and kv head: row r of the block, q head h, chunk c lives at
// part_base + c * stride + (r - row0) * G + (h % G).  nchunks < 0 marks blocks
// whose outputs the tensor-core kernel wrote directly (nothing to combine).
// mblock >= 0 marks a masked row block: nchunks is then only the chunks
// provisioned, and the chunks used come from its list length (masked_chunks
// for `waves` waves of items: 1 on the tensor-core path, kDecListWaves on the
// split-KV path).
struct alignas(16) CombEntry {
  int32_t part_base, nchunks, stride, row0;
  int32_t mblock, waves, pad1, pad2;
};

// Work item of the tensor-core attention kernel: up to NT tiles of 128 query
// vectors (rows [row0, row0 + nrows) of `lane`, G heads each, head-minor
// within a row; tile t holds rows row0 + t*128/G ...) over kv head
// `kv_head`, reading slots [kv_begin, kv_end) in 128-slot KV tiles.  When
// `direct` is set the item covers the rows' whole visible range and writes
// final outputs; otherwise it writes partial softmax states for query q of
// the item at part_base + q (128 per tile).
struct alignas(16) TcItem {
  int32_t lane, kv_head, row0, nrows;
  int32_t kv_begin, kv_end, part_base, direct;
  // masked passes: the row block whose compacted visible-slot list the item
  // walks (else -1), and this item's share of it: chunk `chunk` of `nchunks`
  // equal shares of the list's 128-entry tiles (kv_begin/kv_end unused)
  int32_t block, chunk, nchunks, pad;
};

// A row block of a masked pass: rows [r0, r1) of
// `lane`, whose masks cover nw = ceil(kv_len / 32) words each.  The mask
// pre-pass writes, at these offsets of the scratch arrays, the block's
// compacted list of slots visible to at least one of its rows (list_off, up to
// kv_len entries), and each row's mask re-expressed over that list (cmask_off,
// (r1 - r0) rows of nw words).
struct alignas(16) MaskBlock {
  int32_t lane, r0, r1, nw;
  int32_t list_off, cmask_off, pad0, pad1;
};

constexpr int kStageSlots = 64;   // slots per pipeline stage of the decode kernel
constexpr int kWarpSlots = 16;    // slots per compute warp per stage
constexpr int kTcTileSlots = 128; // slots per KV tile of the tensor-core kernel
constexpr int kTcTileQueries = 128;
// SMs the tensor-core work is sized for when no device is visible (host-only
// planning, e.g. pie_fwd_workspace_bytes on a machine without a GPU); with a
// device, its multiprocessor count is used (device_sm_count).
constexpr int kTcDefaultSms = 152;
int device_sm_count();

// KV slots per tile of the tensor-core kernel with nt query tiles per item
// (two score buffers per query tile and every tile's O share 512 TMEM columns)
constexpr int tc_kv_tile(int nt) { return nt == 1 ? 128 : 64; }

// Chunks a masked unit (row block x kv head) splits its list into: its share
// of one wave of `sms` items (the SMs times the unit's waves), in proportion to its
// KV tiles among all masked units' (total_tiles counts each row block's tiles
// once; every block has Hkv units), at least 1 and at most the provisioned
// items and its tiles.  The kernel and the combine step both use it.
__host__ __device__ inline int masked_chunks(int tiles, int provisioned, int total_tiles, int Hkv,
                                             int sms) {
  if (tiles <= 1) return 1;
  const long long want =
      static_cast<long long>(tiles) * sms / (static_cast<long long>(total_tiles > 0 ? total_tiles : 1) * Hkv);
  long long n = want < 1 ? 1 : want;
  if (n > provisioned) n = provisioned;
  if (n > tiles) n = tiles;
  return static_cast<int>(n);
}

// Device pointers into the caller's workspace, filled by the planner.
struct DevMeta {
  const int32_t* row_indptr;
  const int32_t* positions;
  const int32_t* slots;
  const int32_t* kv_len;
  const int32_t* page_indptr;
  const int32_t* page_ids;
  const int32_t* fold_mode;
  const int32_t* fold_count;
  const int32_t* row_lane;
  const int64_t* mask_word_indptr;  // NULL when the pass has no mask
  const int32_t* readout;
  const int32_t* ro_indptr;         // [N+1]: readout positions of row r are
  const int32_t* ro_idx;            //   ro_idx[ro_indptr[r] .. ro_indptr[r+1])
  const float* rope_freq;           // [d/2]
  const DecItem* dec_items;
  const TcItem* tc_items;
  const CombEntry* comb;            // [row blocks * Hkv]
  const int32_t* row_block;         // [N] row block of each row
  float* part_o;                    // [num_part_slots][d] unnormalised
  float2* part_ml;                  // [num_part_slots] (max, sum), log2 domain
  const MaskBlock* mblocks;         // [num_mblocks] (masked passes whose lanes walk lists)
  int32_t* list;                    // compacted visible-slot lists (scratch)
  int32_t* lrow;                    // page * Hkv * P + slot % P of each listed slot: its
                                    //   row in the pools viewed as [rows][d] is this
                                    //   plus kv_head * P (scratch)
  uint32_t* cmask;                  // rows' masks over the lists (scratch)
  int32_t* list_len;                // [num_mblocks] entries of each list (scratch)
  int32_t* list_mode;               // [num_mblocks] 1: the list is page-granular (scratch)
  int32_t* mask_tiles;              // [1] KV tiles of all masked row blocks' lists (scratch)
  int32_t* dec_work;                // [2] the split-KV items handed out and the CTAs done
                                    //   (zero between launches), or NULL: each CTA walks
                                    //   its fixed run of items
  int32_t num_sms;                  // SMs the masked units' chunks are sized for
  int32_t num_pool_pages;           // page ids at or past it are skipped (PIE_STATUS_BOUNDS)
  int32_t test_stall;               // test hook: 0 none; s + 1: the split-KV producer stops
                                    //   before stage s of every item
  uint32_t test_wait_us;            // test hook: 0, or the split-KV kernel's wait limit in us
};

// Pinned host staging block: metadata uploads copy from pinned memory so that
// they are truly asynchronous.  A released block returns to a process-wide
// pool and is handed out again only once the event recorded after its copy
// has completed.
struct PinnedBlock {
  void* ptr = nullptr;
  size_t cap = 0;
  cudaEvent_t ev = nullptr;
};
PinnedBlock* pinned_acquire(size_t bytes, int* err);
void pinned_release(PinnedBlock* b);

}  // namespace pie

struct pie_fwd_plan {
  pie_fwd_desc desc;
  int32_t L, N, R;
  int32_t G;                 // q heads per kv head
  int32_t num_pool_pages;
  bool has_mask;
  bool any_channel;
  // the combine step's tables (row blocks, combine entries, readout rows) are
  // written by device code of the same stream rather than uploaded with the
  // plan: the combine kernel reads them only after its dependency wait
  bool device_tables;
  int32_t nq;                // query vectors per decode item (2, 4 or 8)
  int32_t num_dec_items;
  int32_t num_tc_items;
  int32_t tc_nt;             // query tiles per tensor-core item (1 or 2)
  int32_t num_mblocks;       // masked row blocks (0 unless some lane walks a list)
  bool dec_lists;            // some split-KV item walks its block's list (the
                             // tensor-core split-KV kernel must take the pass)
  int32_t dec_items_per_cta; // consecutive split-KV items one CTA of the
                             // tensor-core split-KV kernel walks (0 or 1: one)
  int32_t mblock_max_nw;     // largest nw over the masked row blocks
  int32_t mblock_max_rows;   // most rows in a masked row block
  int64_t num_part_slots;
  int32_t num_comb_merge;    // combine entries with chunks to merge (0: no combine launch)
  const uint32_t* mask_set;  // mask words whose compacted lists the workspace holds
                             // (pie_fwd_set_mask), or NULL
  pie::DevMeta dev;
  pie::PinnedBlock* staging;
};

namespace pie {

// Kernel launchers (defined next to their kernels).  Each returns the launch
// status; none synchronizes.
cudaError_t launch_rope_scatter(const pie_fwd_plan_t& p, const void* q, const void* k,
                                const void* v, void* q_rot, void* k_pool, void* v_pool,
                                const int32_t* frozen_len, uint32_t* status, cudaStream_t s);
cudaError_t launch_fold(const pie_fwd_plan_t& p, int32_t* frozen_len, const int32_t* channel,
                        uint32_t* status, cudaStream_t s);
cudaError_t launch_attend_decode(const pie_fwd_plan_t& p, const void* q_rot, const void* k_pool,
                                 const void* v_pool, const uint32_t* mask_words,
                                 uint32_t* status, cudaStream_t s);
// the tensor-core (warp-level MMA) variant of the split-KV kernel, for bf16
// pools with head_dim 128; launch_attend_decode takes it when supported
bool decode_mma_supported(const pie_fwd_plan_t& p);
cudaError_t launch_attend_decode_mma(const pie_fwd_plan_t& p, const void* q_rot,
                                     const void* k_pool, const void* v_pool,
                                     const uint32_t* mask_words, uint32_t* status,
                                     cudaStream_t s);
cudaError_t launch_attend_tc(const pie_fwd_plan_t& p, const void* q_rot, const void* k_pool,
                             const void* v_pool, const uint32_t* mask_words, void* out_readout,
                             float* lse_readout, void* out_all, float* lse_all, uint32_t* status,
                             cudaStream_t s);
cudaError_t launch_mask_compact(const pie_fwd_plan_t& p, const uint32_t* mask_words,
                                cudaStream_t s);
cudaError_t launch_combine(const pie_fwd_plan_t& p, void* out_readout, float* lse_readout,
                           void* out_all, float* lse_all, cudaStream_t s);

// Records `msg` as the calling thread's last error (pie_fwd_last_error) and
// returns `code`.
int set_last_error(int code, const std::string& msg);
// The calling thread's timing events of pie_fwd_set_timing_events (both NULL
// when the hook is off).
void timing_events(cudaEvent_t* start, cudaEvent_t* stop);
// The calling thread's wait-expiry test hook (pie_fwd_test_wait_expiry): the
// stage before which the split-KV producer stops (0: none, else stage + 1) and
// the wait limit in microseconds (0: the default).
void test_wait_hook(int32_t* stall, uint32_t* wait_us);

}  // namespace pie
