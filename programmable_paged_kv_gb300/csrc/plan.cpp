// Host side of the ForwardPass hot path: metadata validation, work-list
// construction, workspace layout, the pinned staging pool and the C entry
// points declared in include/pie_fwd.h.
//
// The planner turns the pass description of the Pie "The forward pass" page
// (lanes by row indptr; StateGeometry positions / slots / kv_len / fold; a
// per-row slot mask; readout rows) into flat device arrays plus two work
// lists:
//   * split-KV items for lanes with few query vectors per kv head (decode,
//     short drafts): each reads one chunk of the lane's slots for up to NQ
//     query vectors;
//   * tensor-core items for lanes with many query vectors (prefill, long
//     drafts, masked prefill): each covers up to 128 query vectors.
// Both kinds leave a partial softmax state (max, sum, unnormalised output)
// per query vector and chunk; a combine step merges the chunks and gathers
// the readout rows.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

namespace pie {

// ---------------------------------------------------------------------------
// errors
// ---------------------------------------------------------------------------
static thread_local std::string g_last_error;

static int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int set_last_error(int code, const std::string& msg) { return fail(code, msg); }

// ---------------------------------------------------------------------------
// pinned staging pool: plans copy their metadata from pinned host memory so
// that the copy is truly asynchronous; a block returns to the pool when its
// plan is destroyed and is reused only after its copy event has completed.
// ---------------------------------------------------------------------------
static std::mutex g_pool_mu;
static std::vector<PinnedBlock*> g_pool_free;

PinnedBlock* pinned_acquire(size_t bytes, int* err) {
  *err = PIE_OK;
  {
    std::lock_guard<std::mutex> lk(g_pool_mu);
    for (size_t i = 0; i < g_pool_free.size(); ++i) {
      PinnedBlock* b = g_pool_free[i];
      if (b->cap >= bytes && cudaEventQuery(b->ev) == cudaSuccess) {
        g_pool_free.erase(g_pool_free.begin() + i);
        return b;
      }
    }
  }
  (void)cudaGetLastError();  // cudaEventQuery may have left cudaErrorNotReady
  size_t cap = 64 << 10;
  while (cap < bytes) cap <<= 1;
  PinnedBlock* b = new PinnedBlock;
  if (cudaMallocHost(&b->ptr, cap) != cudaSuccess) {
    delete b;
    *err = fail(PIE_ECUDA, "cudaMallocHost failed for metadata staging");
    return nullptr;
  }
  if (cudaEventCreateWithFlags(&b->ev, cudaEventDisableTiming) != cudaSuccess) {
    cudaFreeHost(b->ptr);
    delete b;
    *err = fail(PIE_ECUDA, "cudaEventCreate failed for metadata staging");
    return nullptr;
  }
  b->cap = cap;
  return b;
}

void pinned_release(PinnedBlock* b) {
  if (!b) return;
  std::lock_guard<std::mutex> lk(g_pool_mu);
  g_pool_free.push_back(b);
}

// ---------------------------------------------------------------------------
// host plan: validated metadata + work lists, before layout
// ---------------------------------------------------------------------------
struct HostPlan {
  int L = 0, N = 0, R = 0, G = 1, nq = 4, tc_nt = 1, sms = kTcDefaultSms;
  std::vector<int32_t> ro_indptr, ro_idx;
  std::vector<MaskBlock> mblocks;
  int64_t list_total = 0, cmask_total = 0;
  int mblock_max_nw = 0, mblock_max_rows = 0;
  bool has_mask = false, any_channel = false;
  bool dec_lists = false;  // some split-KV item walks a compacted list
  std::vector<int32_t> row_lane, readout;
  std::vector<float> rope_freq;
  std::vector<DecItem> dec;
  std::vector<TcItem> tc;
  std::vector<CombEntry> comb;
  std::vector<int32_t> row_block;
  int64_t num_part_slots = 0;
  int32_t num_comb_merge = 0;
  int64_t total_pages = 0;
};

static bool supported_shape(const pie_fwd_desc& d) {
  return (d.head_dim == 64 || d.head_dim == 128) &&
         (d.page_size == 8 || d.page_size == 16 || d.page_size == 32) &&
         (d.dtype == PIE_F32 || d.dtype == PIE_BF16);
}

static int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// Chunk length (slots, multiple of kStageSlots) for split-KV items.  The
// target keeps several waves of CTAs on a ~150-SM part so that lanes of
// uneven length balance out, without making chunks so short that the
// per-item prologue and the combine traffic dominate.
static int choose_chunk(int64_t total_slots_x_heads) {
  const int64_t kTargetItems = 2048;
  int64_t ch = (total_slots_x_heads + kTargetItems - 1) / kTargetItems;
  ch = std::max<int64_t>(ch, 256);
  ch = std::min<int64_t>(ch, 4096);
  ch = (ch + kTcTileSlots - 1) / kTcTileSlots * kTcTileSlots;  // whole tiles of both kernels
  return static_cast<int>(ch);
}

// Lanes with at least this many query vectors per kv head use the
// tensor-core kernel (bf16 only).
constexpr int kTcMinQueries = 16;

// Multiprocessors of the current device, looked up once per device; the
// default when no device is visible (planning on a host without a GPU).
int device_sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    (void)cudaGetLastError();
    return kTcDefaultSms;
  }
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
    (void)cudaGetLastError();
    return kTcDefaultSms;
  }
  cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

static int build_host_plan(const pie_fwd_desc* desc, const pie_fwd_meta* meta, HostPlan& H) {
  if (!desc || !meta) return fail(PIE_EINVAL, "desc and meta are required");
  const pie_fwd_desc& D = *desc;
  const pie_fwd_meta& M = *meta;
  if (D.num_q_heads <= 0 || D.num_kv_heads <= 0 || D.head_dim <= 0 || D.page_size <= 0)
    return fail(PIE_EINVAL, "head counts, head_dim and page_size must be positive");
  if (D.num_q_heads % D.num_kv_heads != 0)
    return fail(PIE_EINVAL, "num_q_heads must be a multiple of num_kv_heads");
  if (D.dtype != PIE_F32 && D.dtype != PIE_BF16) return fail(PIE_EINVAL, "unknown dtype");
  if (!supported_shape(D))
    return fail(PIE_EUNSUPPORTED, "head_dim must be 64 or 128 and page_size 8, 16 or 32");
  const int G = D.num_q_heads / D.num_kv_heads;
  if (G > 8) return fail(PIE_EUNSUPPORTED, "more than 8 q heads per kv head is not built");
  if (!(D.rope_base > 0.0f)) return fail(PIE_EINVAL, "rope_base must be positive");

  const int L = M.num_lanes, N = M.num_rows;
  if (L < 0 || N < 0 || M.num_pool_pages < 0)
    return fail(PIE_EINVAL, "negative lane, row or pool-page count");
  if (!M.row_indptr || !M.kv_len || !M.page_indptr || !M.fold_mode)
    return fail(PIE_EINVAL, "row_indptr, kv_len, page_indptr and fold_mode are required");
  if (N > 0 && (!M.positions || !M.slots)) return fail(PIE_EINVAL, "positions/slots missing");
  if (M.row_indptr[0] != 0 || M.row_indptr[L] != N)
    return fail(PIE_EINVAL, "row_indptr must start at 0 and end at num_rows");
  if (M.page_indptr[0] != 0) return fail(PIE_EINVAL, "page_indptr must start at 0");
  for (int l = 0; l < L; ++l) {
    if (M.row_indptr[l + 1] < M.row_indptr[l]) return fail(PIE_EINVAL, "row_indptr decreases");
    if (M.page_indptr[l + 1] < M.page_indptr[l]) return fail(PIE_EINVAL, "page_indptr decreases");
  }
  const int64_t total_pages = M.page_indptr[L];
  if (total_pages > 0 && !M.page_ids) return fail(PIE_EINVAL, "page_ids missing");
  {
    // range of the page ids (one branch-free pass the compiler vectorizes)
    int32_t lo = 0, hi = 0;
    if (total_pages > 0) lo = hi = M.page_ids[0];
    for (int64_t i = 0; i < total_pages; ++i) {
      lo = std::min(lo, M.page_ids[i]);
      hi = std::max(hi, M.page_ids[i]);
    }
    if (total_pages > 0 && (lo < 0 || hi >= M.num_pool_pages))
      return fail(PIE_ERANGE, "page id outside the pool");
  }

  H.L = L;
  H.N = N;
  H.G = G;
  H.sms = device_sm_count();
  H.total_pages = total_pages;
  H.row_lane.assign(N, 0);
  H.any_channel = false;
  int max_rows = 0;
  for (int l = 0; l < L; ++l) {
    const int r0 = M.row_indptr[l], r1 = M.row_indptr[l + 1], n = r1 - r0;
    max_rows = std::max(max_rows, n);
    const int64_t cap = static_cast<int64_t>(M.page_indptr[l + 1] - M.page_indptr[l]) * D.page_size;
    if (M.kv_len[l] < 0 || M.kv_len[l] > cap) return fail(PIE_ERANGE, "kv_len outside the lane's pages");
    for (int r = r0; r < r1; ++r) {
      H.row_lane[r] = l;
      if (M.positions[r] < 0) return fail(PIE_ERANGE, "negative position");
      if (M.slots[r] < 0 || M.slots[r] >= cap) return fail(PIE_ERANGE, "slot outside the lane's pages");
    }
    const int fm = M.fold_mode[l];
    if (fm < PIE_FOLD_NONE || fm > PIE_FOLD_CHANNEL) return fail(PIE_EINVAL, "unknown fold mode");
    if (fm == PIE_FOLD_COUNT) {
      if (!M.fold_count) return fail(PIE_EINVAL, "fold_count missing");
      if (M.fold_count[l] < 0 || M.fold_count[l] > n) return fail(PIE_ERANGE, "fold_count outside [0, n]");
    }
    if (fm == PIE_FOLD_CHANNEL) H.any_channel = true;
    if (fm != PIE_FOLD_NONE)
      for (int r = r0 + 1; r < r1; ++r)
        if (M.slots[r] != M.slots[r - 1] + 1)
          return fail(PIE_EINVAL, "a folding lane must write consecutive slots");
  }
  // Hazard freedom (Pie review, Eq. (4)): the rows of one pass write
  // pairwise distinct physical slots.
  // Checked with an open-addressing hash set of the physical targets
  // (linear time; the table is reused across plans on a thread).
  {
    static thread_local std::vector<int64_t> table;
    int bits = 6;
    while ((int64_t(1) << bits) < 2 * static_cast<int64_t>(N)) ++bits;
    const size_t size = size_t(1) << bits;
    if (table.size() < size) table.resize(size);
    std::fill(table.begin(), table.begin() + size, int64_t(-1));
    for (int r = 0; r < N; ++r) {
      const int l = H.row_lane[r], s = M.slots[r];
      const int64_t page = M.page_ids[M.page_indptr[l] + s / D.page_size];
      const int64_t key = page * D.page_size + s % D.page_size;
      size_t h = static_cast<size_t>((static_cast<uint64_t>(key) * 0x9E3779B97F4A7C15ull) >> (64 - bits));
      while (table[h] != -1) {
        if (table[h] == key) return fail(PIE_EINVAL, "two rows write the same physical slot");
        h = (h + 1) & (size - 1);
      }
      table[h] = key;
    }
  }
  H.has_mask = M.mask_word_indptr != nullptr;
  if (H.has_mask) {
    if (M.mask_word_indptr[0] != 0) return fail(PIE_EINVAL, "mask_word_indptr must start at 0");
    for (int r = 0; r < N; ++r) {
      const int64_t nw = M.mask_word_indptr[r + 1] - M.mask_word_indptr[r];
      if (nw < 0) return fail(PIE_EINVAL, "mask_word_indptr decreases");
      if (nw < (static_cast<int64_t>(M.kv_len[H.row_lane[r]]) + 31) / 32)
        return fail(PIE_ERANGE, "a row has fewer than ceil(kv_len/32) mask words");
    }
  }
  H.readout.clear();
  if (M.readout) {
    if (M.num_readout < 0) return fail(PIE_EINVAL, "negative num_readout");
    for (int j = 0; j < M.num_readout; ++j) {
      if (M.readout[j] < 0 || M.readout[j] >= N) return fail(PIE_ERANGE, "readout row out of range");
      H.readout.push_back(M.readout[j]);
    }
  } else {
    for (int l = 0; l < L; ++l)
      if (M.row_indptr[l + 1] > M.row_indptr[l]) H.readout.push_back(M.row_indptr[l + 1] - 1);
  }
  H.R = static_cast<int>(H.readout.size());

  // RoPE frequencies base^(-2i/d), computed in double, rounded once to float.
  const int d = D.head_dim;
  H.rope_freq.resize(d / 2);
  for (int i = 0; i < d / 2; ++i)
    H.rope_freq[i] = static_cast<float>(std::pow(static_cast<double>(D.rope_base), -2.0 * i / d));

  // ---- work lists ---------------------------------------------------------
  const int Hkv = D.num_kv_heads;
  // query vectors per split-KV item: a whole GQA group of as many rows as
  // fit in 8 vectors, at least 2 (the kernel's reduction needs 2)
  const int rows_fit = std::max(1, std::min(max_rows, 8 / G));
  H.nq = std::min(8, std::max(2, next_pow2(G * rows_fit)));
  const int rows_per_item = std::max(1, H.nq / G);
  // the kv extent a block of rows needs: causal => up to its last slot + 1
  auto extent = [&](int l, int r0, int r1) {
    const int kv = M.kv_len[l];
    if (H.has_mask) return kv;
    int mx = -1;
    for (int r = r0; r < r1; ++r) mx = std::max(mx, M.slots[r]);
    return std::min(kv, mx + 1);
  };
  // (the tensor-core kernel addresses pool rows with 32-bit TMA coordinates)
  const bool tc_ok = D.dtype == PIE_BF16 && D.head_dim == 128 &&
                     kTcTileQueries % G == 0 &&
                     static_cast<int64_t>(M.num_pool_pages) * Hkv * D.page_size <= INT32_MAX;
  // the tensor-core split-KV kernel (bf16, d 128, 32-bit tensor-copy rows);
  // the launch takes it under the same condition (decode_mma_supported)
  const int64_t pool_rows = static_cast<int64_t>(M.num_pool_pages) * Hkv * D.page_size;
  const bool mma_ok = D.dtype == PIE_BF16 && D.head_dim == 128 && pool_rows > 0 &&
                      pool_rows <= INT32_MAX;
  // Lanes with many query vectors per kv head go to the tensor-core kernel.  In
  // a masked pass both kernels walk the compacted list of the slots a row
  // block sees (whole pages of a window, single rows of a scattered mask), so a
  // masked row reads only what it attends; a masked lane the list-walking
  // kernels cannot take (fp32, d 64) reads its whole range on the scalar
  // split-KV kernel.
  auto lane_tc = [&](int l) {
    const int n = M.row_indptr[l + 1] - M.row_indptr[l];
    return tc_ok && n > 0 && (n * G >= kTcMinQueries || (H.has_mask && !mma_ok));
  };
  auto lane_list = [&](int l) { return H.has_mask && (lane_tc(l) || mma_ok); };
  // split-KV items: chunk length from the total work
  int64_t work = 0;
  for (int l = 0; l < L; ++l)
    if (!lane_tc(l)) work += static_cast<int64_t>(M.kv_len[l]) * Hkv;
  const int CH = choose_chunk(work);
  // tensor-core items: two query tiles per item when some lane has more than
  // 128 query vectors per kv head (they then share every K/V tile)
  int max_tc_q = 0;
  for (int l = 0; l < L; ++l)
    if (lane_tc(l)) max_tc_q = std::max(max_tc_q, (M.row_indptr[l + 1] - M.row_indptr[l]) * G);
  H.tc_nt = max_tc_q > kTcTileQueries ? 2 : 1;
  const int tc_rows = std::max(1, H.tc_nt * kTcTileQueries / G);
  // split a tensor-core unit's KV range only as far as needed to give about
  // four waves of items; the nearest whole number of chunks, each a whole
  // number of 128-slot tiles
  int64_t tc_total = 0, tc_units = 0;
  for (int l = 0; l < L; ++l) {
    if (!lane_tc(l)) continue;
    const int r0 = M.row_indptr[l], r1 = M.row_indptr[l + 1];
    for (int b0 = r0; b0 < r1; b0 += tc_rows) {
      tc_total += static_cast<int64_t>(extent(l, b0, std::min(r1, b0 + tc_rows))) * Hkv;
      tc_units += Hkv;
    }
  }
  const int64_t tc_target = 4 * static_cast<int64_t>(H.sms);
  const int64_t tc_ch = tc_units >= tc_target ? INT32_MAX
                        : std::max<int64_t>(512, (tc_total + tc_target - 1) / tc_target);
  H.comb.clear();
  H.num_comb_merge = 0;
  H.row_block.assign(N, 0);
  H.dec.clear();
  H.tc.clear();
  // masked passes: the list-walking lanes' items walk the compacted list of
  // the slots their row block can see (one list per row block, shared by all
  // kv heads)
  H.mblocks.clear();
  bool any_list = false;
  for (int l = 0; l < L; ++l) any_list = any_list || lane_list(l);
  std::vector<int32_t> block_of_row(any_list ? N : 0, -1);
  H.list_total = H.cmask_total = 0;
  H.mblock_max_nw = H.mblock_max_rows = 0;
  H.dec_lists = false;
  if (!block_of_row.empty()) {
    for (int l = 0; l < L; ++l) {
      if (!lane_list(l)) continue;
      const int r0 = M.row_indptr[l], r1 = M.row_indptr[l + 1];
      const int nw = (M.kv_len[l] + 31) / 32;
      const int blk_rows = lane_tc(l) ? tc_rows : rows_per_item;
      H.dec_lists = H.dec_lists || (!lane_tc(l) && r1 > r0);
      for (int b0 = r0; b0 < r1; b0 += blk_rows) {
        const int b1 = std::min(r1, b0 + blk_rows);
        block_of_row[b0] = static_cast<int32_t>(H.mblocks.size());
        H.mblocks.push_back(MaskBlock{l, b0, b1, nw, static_cast<int32_t>(H.list_total),
                                      static_cast<int32_t>(H.cmask_total), 0, 0});
        H.list_total += M.kv_len[l];
        H.cmask_total += static_cast<int64_t>(b1 - b0) * nw;
        H.mblock_max_nw = std::max(H.mblock_max_nw, nw);
        H.mblock_max_rows = std::max(H.mblock_max_rows, b1 - b0);
      }
    }
    if (H.list_total > INT32_MAX || H.cmask_total > INT32_MAX)
      return fail(PIE_ERANGE, "masked pass too large for the compacted slot lists");
  }
  int64_t part = 0;
  for (int l = 0; l < L; ++l) {
    const int r0 = M.row_indptr[l], r1 = M.row_indptr[l + 1], n = r1 - r0;
    if (n == 0) continue;
    const bool use_tc = lane_tc(l);
    const int blk_rows = use_tc ? tc_rows : rows_per_item;
    const int stride = use_tc ? kTcTileQueries : H.nq;
    for (int b0 = r0; b0 < r1; b0 += blk_rows) {
      const int b1 = std::min(r1, b0 + blk_rows);
      const int32_t blk_id = static_cast<int32_t>(H.comb.size() / Hkv);
      for (int r = b0; r < b1; ++r) H.row_block[r] = blk_id;
      const int ext = extent(l, b0, b1);
      int nchunks, chunk;
      if (use_tc) {
        nchunks = static_cast<int>(std::max<int64_t>(1, (ext + tc_ch / 2) / tc_ch));
        chunk = ((ext + nchunks - 1) / nchunks + kTcTileSlots - 1) / kTcTileSlots * kTcTileSlots;
        nchunks = std::max(1, (ext + chunk - 1) / std::max(1, chunk));
      } else {
        // a listed unit has at least one item: the combine step reads at
        // least one chunk of every list (an empty list's item writes the
        // empty state)
        nchunks = (ext + CH - 1) / CH;
        if (!block_of_row.empty() && block_of_row[b0] >= 0) nchunks = std::max(1, nchunks);
        chunk = CH;
      }
      const bool direct = use_tc && nchunks == 1;
      const int32_t mblk = block_of_row.empty() ? -1 : block_of_row[b0];
      for (int g = 0; g < Hkv; ++g) {
        H.comb.push_back(CombEntry{static_cast<int32_t>(part), direct ? -1 : nchunks,
                                   use_tc ? stride * H.tc_nt : stride, b0, mblk,
                                   use_tc ? 1 : kDecListWaves, 0, 0});
        if (!direct) ++H.num_comb_merge;
        if (use_tc) {
          for (int c = 0; c < nchunks; ++c) {
            const int kb = c * chunk, ke = std::min(ext, kb + chunk);
            H.tc.push_back(TcItem{l, g, b0, b1 - b0, kb, ke, static_cast<int32_t>(part),
                                  direct ? 1 : 0, mblk, c, nchunks, 0});
            part += direct ? 0 : stride * H.tc_nt;
          }
        } else {
          // the unit's chunks written in place (a decode batch has thousands);
          // a listed item names its list block and its chunk of the list
          const size_t base = H.dec.size();
          H.dec.resize(base + nchunks);
          DecItem* di = H.dec.data() + base;
          for (int c = 0; c < nchunks; ++c) {
            const int kb = c * chunk;
            const int32_t pb = static_cast<int32_t>(part + int64_t(c) * stride);
            di[c] = mblk >= 0 ? DecItem{l, g, b0, b1 - b0, c, nchunks, pb, mblk}
                              : DecItem{l, g, b0, b1 - b0, kb, std::min(ext, kb + chunk), pb, -1};
          }
          part += int64_t(nchunks) * stride;
        }
      }
    }
  }
  // listed split-KV items chunk-major (every unit's first chunk, then every
  // unit's second, ...): the CTAs in flight spread over all lanes and kv
  // heads, and the chunks a short list leaves unused come last
  if (H.dec_lists)
    std::stable_sort(H.dec.begin(), H.dec.end(), [](const DecItem& a, const DecItem& b) {
      return (a.block >= 0 ? a.kv_begin : 0) < (b.block >= 0 ? b.kv_begin : 0);
    });
  // readout positions per row (a row may be read out several times)
  H.ro_indptr.assign(N + 1, 0);
  for (int j = 0; j < H.R; ++j) H.ro_indptr[H.readout[j] + 1]++;
  for (int r = 0; r < N; ++r) H.ro_indptr[r + 1] += H.ro_indptr[r];
  H.ro_idx.assign(H.R, 0);
  {
    std::vector<int32_t> fill(H.ro_indptr.begin(), H.ro_indptr.end() - 1);
    for (int j = 0; j < H.R; ++j) H.ro_idx[fill[H.readout[j]]++] = j;
  }
  if (part > INT32_MAX) return fail(PIE_ERANGE, "pass too large: partial index overflow");
  H.num_part_slots = part;
  return PIE_OK;
}

// ---------------------------------------------------------------------------
// workspace layout: metadata and work lists (copied from the host), then
// the partials (device scratch).
// ---------------------------------------------------------------------------
struct Layout {
  size_t row_indptr, positions, slots, kv_len, page_indptr, page_ids, fold_mode, fold_count,
      row_lane, mask_word_indptr, readout, ro_indptr, ro_idx, rope_freq, dec, tc, comb, mblocks,
      row_block;
  size_t copy_bytes;  // everything above
  size_t part_o, part_ml, list, lrow, cmask, list_len, list_mode, mask_tiles, dec_work;
  size_t total;
};

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

static Layout make_layout(const pie_fwd_desc& D, const HostPlan& H) {
  Layout Y{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  Y.row_indptr = take(4 * (H.L + 1));
  Y.positions = take(4 * H.N);
  Y.slots = take(4 * H.N);
  Y.kv_len = take(4 * H.L);
  Y.page_indptr = take(4 * (H.L + 1));
  Y.page_ids = take(4 * H.total_pages);
  Y.fold_mode = take(4 * H.L);
  Y.fold_count = take(4 * H.L);
  Y.row_lane = take(4 * H.N);
  Y.mask_word_indptr = take(H.has_mask ? 8 * (H.N + 1) : 0);
  Y.readout = take(4 * H.R);
  Y.ro_indptr = take(4 * (H.N + 1));
  Y.ro_idx = take(4 * H.R);
  Y.rope_freq = take(4 * (D.head_dim / 2));
  Y.dec = take(sizeof(DecItem) * H.dec.size());
  Y.tc = take(sizeof(TcItem) * H.tc.size());
  Y.comb = take(sizeof(CombEntry) * H.comb.size());
  Y.row_block = take(sizeof(int32_t) * H.row_block.size());
  Y.mblocks = take(sizeof(MaskBlock) * H.mblocks.size());
  // the split-KV kernel's work counter and finished-CTA count (zero from the
  // upload; the kernel sets them back to zero when it ends)
  Y.dec_work = take(H.dec.empty() ? 0 : 2 * sizeof(int32_t));
  Y.copy_bytes = o;
  Y.part_o = take(sizeof(float) * static_cast<size_t>(H.num_part_slots) * D.head_dim);
  Y.part_ml = take(sizeof(float2) * static_cast<size_t>(H.num_part_slots));
  Y.list = take(sizeof(int32_t) * static_cast<size_t>(H.list_total));
  Y.lrow = take(sizeof(int32_t) * static_cast<size_t>(H.list_total));
  Y.cmask = take(sizeof(uint32_t) * static_cast<size_t>(H.cmask_total));
  Y.list_len = take(sizeof(int32_t) * H.mblocks.size());
  Y.list_mode = take(sizeof(int32_t) * H.mblocks.size());
  Y.mask_tiles = take(H.mblocks.empty() ? 0 : sizeof(int32_t));
  Y.total = o;
  return Y;
}

}  // namespace pie

using namespace pie;

extern "C" {

const char* pie_fwd_last_error(void) { return g_last_error.c_str(); }

int pie_fwd_abi_version(void) { return 105; }

static thread_local cudaEvent_t g_ev_start = nullptr, g_ev_stop = nullptr;

int pie_fwd_set_timing_events(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr))
    return fail(PIE_EINVAL, "timing events: give both or neither");
  g_ev_start = static_cast<cudaEvent_t>(start_event);
  g_ev_stop = static_cast<cudaEvent_t>(stop_event);
  return PIE_OK;
}

}  // extern "C"

void pie::timing_events(cudaEvent_t* start, cudaEvent_t* stop) {
  *start = g_ev_start;
  *stop = g_ev_stop;
}

static thread_local int32_t g_test_stall = 0;
static thread_local uint32_t g_test_wait_us = 0;

extern "C" int pie_fwd_test_wait_expiry(int32_t stage, uint32_t wait_us) {
  if (stage < -1) return fail(PIE_EINVAL, "test_wait_expiry: stage must be -1 or >= 0");
  if (stage >= 0 && wait_us == 0) return fail(PIE_EINVAL, "test_wait_expiry: give a wait limit");
  g_test_stall = stage + 1;
  g_test_wait_us = stage >= 0 ? wait_us : 0;
  return PIE_OK;
}

void pie::test_wait_hook(int32_t* stall, uint32_t* wait_us) {
  *stall = g_test_stall;
  *wait_us = g_test_wait_us;
}

extern "C" {

// One host plan per calling thread, reused so that its vectors keep their
// capacity from one pass to the next (build_host_plan resets every field).
static HostPlan& thread_host_plan() {
  static thread_local HostPlan H;
  return H;
}

int pie_fwd_workspace_bytes(const pie_fwd_desc* desc, const pie_fwd_meta* meta, size_t* bytes) {
  if (!bytes) return fail(PIE_EINVAL, "bytes is NULL");
  HostPlan& H = thread_host_plan();
  int rc = build_host_plan(desc, meta, H);
  if (rc != PIE_OK) return rc;
  *bytes = make_layout(*desc, H).total;
  return PIE_OK;
}

int pie_fwd_plan(const pie_fwd_desc* desc, const pie_fwd_meta* meta, void* dev_workspace,
                 size_t ws_bytes, void* stream, pie_fwd_plan_t** out) {
  if (!out) return fail(PIE_EINVAL, "out is NULL");
  *out = nullptr;
  HostPlan& H = thread_host_plan();
  int rc = build_host_plan(desc, meta, H);
  if (rc != PIE_OK) return rc;
  const pie_fwd_meta& M = *meta;
  Layout Y = make_layout(*desc, H);
  if (ws_bytes < Y.total || (Y.total > 0 && !dev_workspace))
    return fail(PIE_ENOSPACE, "workspace smaller than pie_fwd_workspace_bytes()");
  if (reinterpret_cast<uintptr_t>(dev_workspace) % 256 != 0)
    return fail(PIE_EINVAL, "workspace must be 256-byte aligned");

  int err = PIE_OK;
  PinnedBlock* blk = pinned_acquire(std::max<size_t>(Y.copy_bytes, 1), &err);
  if (!blk) return err;
  char* h = static_cast<char*>(blk->ptr);
  std::memset(h, 0, Y.copy_bytes);
  auto put = [&](size_t off, const void* src, size_t bytes) {
    if (bytes) std::memcpy(h + off, src, bytes);
  };
  put(Y.row_indptr, M.row_indptr, 4 * (H.L + 1));
  put(Y.positions, M.positions, 4 * H.N);
  put(Y.slots, M.slots, 4 * H.N);
  put(Y.kv_len, M.kv_len, 4 * H.L);
  put(Y.page_indptr, M.page_indptr, 4 * (H.L + 1));
  put(Y.page_ids, M.page_ids, 4 * H.total_pages);
  put(Y.fold_mode, M.fold_mode, 4 * H.L);
  if (M.fold_count) put(Y.fold_count, M.fold_count, 4 * H.L);
  put(Y.row_lane, H.row_lane.data(), 4 * H.N);
  if (H.has_mask) put(Y.mask_word_indptr, M.mask_word_indptr, 8 * (H.N + 1));
  put(Y.readout, H.readout.data(), 4 * H.R);
  put(Y.ro_indptr, H.ro_indptr.data(), 4 * (H.N + 1));
  put(Y.ro_idx, H.ro_idx.data(), 4 * H.R);
  put(Y.rope_freq, H.rope_freq.data(), 4 * H.rope_freq.size());
  put(Y.dec, H.dec.data(), sizeof(DecItem) * H.dec.size());
  put(Y.tc, H.tc.data(), sizeof(TcItem) * H.tc.size());
  put(Y.comb, H.comb.data(), sizeof(CombEntry) * H.comb.size());
  put(Y.row_block, H.row_block.data(), sizeof(int32_t) * H.row_block.size());
  put(Y.mblocks, H.mblocks.data(), sizeof(MaskBlock) * H.mblocks.size());

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (Y.copy_bytes > 0 &&
      cudaMemcpyAsync(dev_workspace, h, Y.copy_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
    pinned_release(blk);
    return fail(PIE_ECUDA, std::string("plan upload failed: ") + cudaGetErrorString(cudaGetLastError()));
  }
  if (cudaEventRecord(blk->ev, s) != cudaSuccess) {
    // the copy is queued; keep the block out of the pool rather than risk reuse
    return fail(PIE_ECUDA, "cudaEventRecord failed after the plan upload");
  }

  pie_fwd_plan_t* p = new pie_fwd_plan_t;
  std::memset(p, 0, sizeof(*p));
  p->desc = *desc;
  if (p->desc.sm_scale == 0.0f) p->desc.sm_scale = 1.0f / std::sqrt(static_cast<float>(desc->head_dim));
  p->L = H.L;
  p->N = H.N;
  p->R = H.R;
  p->G = H.G;
  p->num_pool_pages = M.num_pool_pages;
  p->has_mask = H.has_mask;
  p->any_channel = H.any_channel;
  p->nq = H.nq;
  p->num_dec_items = static_cast<int32_t>(H.dec.size());
  p->num_tc_items = static_cast<int32_t>(H.tc.size());
  p->tc_nt = H.tc_nt;
  p->num_mblocks = static_cast<int32_t>(H.mblocks.size());
  p->dec_lists = H.dec_lists;
  p->dec_items_per_cta = H.dec_lists ? kDecListItemsPerCta : 1;
  p->mblock_max_nw = H.mblock_max_nw;
  p->mblock_max_rows = H.mblock_max_rows;
  p->num_part_slots = H.num_part_slots;
  p->num_comb_merge = H.num_comb_merge;
  char* w = static_cast<char*>(dev_workspace);
  DevMeta& dm = p->dev;
  dm.row_indptr = reinterpret_cast<const int32_t*>(w + Y.row_indptr);
  dm.positions = reinterpret_cast<const int32_t*>(w + Y.positions);
  dm.slots = reinterpret_cast<const int32_t*>(w + Y.slots);
  dm.kv_len = reinterpret_cast<const int32_t*>(w + Y.kv_len);
  dm.page_indptr = reinterpret_cast<const int32_t*>(w + Y.page_indptr);
  dm.page_ids = reinterpret_cast<const int32_t*>(w + Y.page_ids);
  dm.fold_mode = reinterpret_cast<const int32_t*>(w + Y.fold_mode);
  dm.fold_count = reinterpret_cast<const int32_t*>(w + Y.fold_count);
  dm.row_lane = reinterpret_cast<const int32_t*>(w + Y.row_lane);
  dm.mask_word_indptr = H.has_mask ? reinterpret_cast<const int64_t*>(w + Y.mask_word_indptr) : nullptr;
  dm.readout = reinterpret_cast<const int32_t*>(w + Y.readout);
  dm.ro_indptr = reinterpret_cast<const int32_t*>(w + Y.ro_indptr);
  dm.ro_idx = reinterpret_cast<const int32_t*>(w + Y.ro_idx);
  dm.rope_freq = reinterpret_cast<const float*>(w + Y.rope_freq);
  dm.dec_items = reinterpret_cast<const DecItem*>(w + Y.dec);
  dm.tc_items = reinterpret_cast<const TcItem*>(w + Y.tc);
  dm.comb = reinterpret_cast<const CombEntry*>(w + Y.comb);
  dm.row_block = reinterpret_cast<const int32_t*>(w + Y.row_block);
  dm.part_o = reinterpret_cast<float*>(w + Y.part_o);
  dm.part_ml = reinterpret_cast<float2*>(w + Y.part_ml);
  dm.mblocks = reinterpret_cast<const MaskBlock*>(w + Y.mblocks);
  dm.list = reinterpret_cast<int32_t*>(w + Y.list);
  dm.lrow = reinterpret_cast<int32_t*>(w + Y.lrow);
  dm.cmask = reinterpret_cast<uint32_t*>(w + Y.cmask);
  dm.list_len = reinterpret_cast<int32_t*>(w + Y.list_len);
  dm.list_mode = reinterpret_cast<int32_t*>(w + Y.list_mode);
  dm.mask_tiles = reinterpret_cast<int32_t*>(w + Y.mask_tiles);
  // plain passes: a persistent grid takes the split-KV items from the counter;
  // list passes: fixed runs of kDecListItemsPerCta items per CTA
  dm.dec_work = (H.dec.empty() || H.dec_lists) ? nullptr
                                                : reinterpret_cast<int32_t*>(w + Y.dec_work);
  dm.num_sms = H.sms;
  dm.num_pool_pages = M.num_pool_pages;
  p->staging = blk;
  *out = p;
  return PIE_OK;
}

int32_t pie_fwd_plan_num_readout(const pie_fwd_plan_t* plan) { return plan ? plan->R : -1; }

void pie_fwd_plan_destroy(pie_fwd_plan_t* plan) {
  if (!plan) return;
  pinned_release(plan->staging);  // reused only after its copy event completes
  delete plan;
}

int pie_fwd_append_kv(const pie_fwd_plan_t* plan, const void* q, const void* k, const void* v,
                      void* q_rot, void* k_pool, void* v_pool, const int32_t* frozen_len,
                      uint32_t* status, void* stream) {
  if (!plan) return fail(PIE_EINVAL, "plan is NULL");
  if (plan->N == 0) return PIE_OK;
  if (!q || !k || !v || !q_rot || !k_pool || !v_pool || !frozen_len)
    return fail(PIE_EINVAL, "append_kv: a required pointer is NULL");
  cudaError_t e = launch_rope_scatter(*plan, q, k, v, q_rot, k_pool, v_pool, frozen_len, status,
                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(PIE_ECUDA, std::string("append_kv launch: ") + cudaGetErrorString(e));
  return PIE_OK;
}

int pie_fwd_attend(const pie_fwd_plan_t* plan, const void* q_rot, const void* k_pool,
                   const void* v_pool, const uint32_t* mask_words, void* out_readout,
                   float* lse_readout, void* out_all, float* lse_all, uint32_t* status,
                   void* stream) {
  if (!plan) return fail(PIE_EINVAL, "plan is NULL");
  if (plan->has_mask && !mask_words) return fail(PIE_EINVAL, "the plan has a mask: mask_words required");
  if (!plan->has_mask && mask_words) return fail(PIE_EINVAL, "mask_words given but the plan has no mask");
  if (plan->N == 0) return PIE_OK;
  if (!q_rot || !k_pool || !v_pool) return fail(PIE_EINVAL, "attend: q_rot and pools are required");
  if (plan->R > 0 && !out_readout && !out_all)
    return fail(PIE_EINVAL, "attend: out_readout (or out_all) is required");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  // the compacted lists are a function of the pass (mask words and page
  // table), not of the layer: after pie_fwd_set_mask they are reused
  if (plan->num_mblocks > 0 && mask_words != plan->mask_set)
    e = launch_mask_compact(*plan, mask_words, s);
  if (e == cudaSuccess && g_ev_start) e = cudaEventRecord(g_ev_start, s);
  if (e == cudaSuccess && plan->num_dec_items > 0)
    e = launch_attend_decode(*plan, q_rot, k_pool, v_pool, mask_words, status, s);
  if (e == cudaSuccess && plan->num_tc_items > 0)
    e = launch_attend_tc(*plan, q_rot, k_pool, v_pool, mask_words, out_readout, lse_readout,
                         out_all, lse_all, status, s);
  if (e == cudaSuccess && g_ev_stop) e = cudaEventRecord(g_ev_stop, s);
  if (e == cudaSuccess && plan->num_comb_merge > 0)
    e = launch_combine(*plan, out_readout, lse_readout, out_all, lse_all, s);
  if (e != cudaSuccess) return fail(PIE_ECUDA, std::string("attend launch: ") + cudaGetErrorString(e));
  return PIE_OK;
}

int pie_fwd_set_mask(pie_fwd_plan_t* plan, const uint32_t* mask_words, void* stream) {
  if (!plan) return fail(PIE_EINVAL, "plan is NULL");
  if (!plan->has_mask) return fail(PIE_EINVAL, "set_mask: the plan has no mask");
  if (!mask_words) return fail(PIE_EINVAL, "set_mask: mask_words is NULL");
  plan->mask_set = nullptr;
  if (plan->num_mblocks > 0) {
    cudaError_t e = launch_mask_compact(*plan, mask_words, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
      return fail(PIE_ECUDA, std::string("set_mask launch: ") + cudaGetErrorString(e));
  }
  plan->mask_set = mask_words;
  return PIE_OK;
}

int pie_fwd_forward(const pie_fwd_desc* desc, const pie_fwd_meta* meta, void* dev_workspace,
                    size_t ws_bytes, const void* q, const void* k, const void* v, void* q_rot,
                    void* k_pool, void* v_pool, int32_t* frozen_len, const uint32_t* mask_words,
                    void* out_readout, float* lse_readout, void* out_all, float* lse_all,
                    const int32_t* channel, uint32_t* status, void* stream) {
  pie_fwd_plan_t* plan = nullptr;
  int rc = pie_fwd_plan(desc, meta, dev_workspace, ws_bytes, stream, &plan);
  if (rc != PIE_OK) return rc;
  rc = pie_fwd_append_kv(plan, q, k, v, q_rot, k_pool, v_pool, frozen_len, status, stream);
  if (rc == PIE_OK && plan->has_mask && mask_words) rc = pie_fwd_set_mask(plan, mask_words, stream);
  if (rc == PIE_OK)
    rc = pie_fwd_attend(plan, q_rot, k_pool, v_pool, mask_words, out_readout, lse_readout,
                        out_all, lse_all, status, stream);
  if (rc == PIE_OK) rc = pie_fwd_fold(plan, frozen_len, channel, status, stream);
  pie_fwd_plan_destroy(plan);
  return rc;
}

int pie_fwd_fold(const pie_fwd_plan_t* plan, int32_t* frozen_len, const int32_t* channel,
                 uint32_t* status, void* stream) {
  if (!plan) return fail(PIE_EINVAL, "plan is NULL");
  if (plan->L == 0) return PIE_OK;
  if (!frozen_len) return fail(PIE_EINVAL, "fold: frozen_len is NULL");
  if (plan->any_channel && !channel) return fail(PIE_EINVAL, "fold: a lane folds from the channel");
  cudaError_t e = launch_fold(*plan, frozen_len, channel, status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(PIE_ECUDA, std::string("fold launch: ") + cudaGetErrorString(e));
  return PIE_OK;
}

}  // extern "C"
