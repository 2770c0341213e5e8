// A decode loop that runs ahead of the host (Pie "The forward pass",
// Pipelines and frames: run_ahead keeps a repeating decode pass in flight on
// the GPU; passes on one pipeline run in submission order).
//
// pie_fwd_decode_loop runs `steps` single-row ForwardPasses per lane back to
// back.  Step t of lane l is the folding() geometry of one new token (State
// geometry): position = slot = frozen_len[l], kv_len = frozen_len[l] + 1,
// fold all.  The geometry and the split-KV work items come from frozen_len on
// the device, so no host plan is built per token and the whole call -- a
// handful of launches per step, no host synchronization, no allocation -- can
// be captured in a CUDA graph by the caller.  Each step reuses the pass
// kernels: RoPE + slot scatter, split-KV attention, combine into out[t],
// fold.
//
// A lane whose pages hold no slot for its next token (frozen_len[l] >= its
// pages x page_size) writes nothing, gets a zero output and -inf lse, does not
// advance, and sets PIE_STATUS_LOOP_FULL.
//
// With a channel (device int32 [steps][L]), step t freezes clamp(channel[t][l],
// 0, 1) slots instead of one (State geometry, speculative-decoding paragraph:
// the count comes from a device channel; a count outside [0, 1] is clamped and
// sets PIE_STATUS_FOLD_CLAMP).  A lane whose count is 0 keeps its frozen
// length: its next step writes the same slot again, at the same position, so
// the rejected token's K/V is overwritten before anything reads it.  Whatever
// device code decides the counts (a stop-token test, a draft acceptance) writes
// channel[t] before step t's fold on the stream.

#include <cmath>
#include <cstring>
#include <string>

#include "common.cuh"

namespace pie {

constexpr int kLoopChunk = 512;  // slots per split-KV item (a multiple of kStageSlots)

struct LoopLayout {
  size_t row_indptr, row_lane, positions, slots, kv_len, fold_mode, fold_count, readout,
      ro_indptr, ro_idx, rope_freq, dec, comb, row_block, work, part_ml, part_o, total;
};

static LoopLayout loop_layout(int L, int Hkv, int MC, int nq, int d) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  LoopLayout Y{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = al(o + bytes);
    return at;
  };
  const size_t Ls = static_cast<size_t>(L), items = Ls * Hkv * MC;
  Y.row_indptr = take(4 * (Ls + 1));
  Y.row_lane = take(4 * Ls);
  Y.positions = take(4 * Ls);
  Y.slots = take(4 * Ls);
  Y.kv_len = take(4 * Ls);
  Y.fold_mode = take(4 * Ls);
  Y.fold_count = take(4 * Ls);
  Y.readout = take(4 * Ls);
  Y.ro_indptr = take(4 * (Ls + 1));
  Y.ro_idx = take(4 * Ls);
  Y.rope_freq = take(4 * static_cast<size_t>(d / 2));
  Y.dec = take(sizeof(DecItem) * items);
  Y.comb = take(sizeof(CombEntry) * Ls * Hkv);
  Y.row_block = take(4 * Ls);
  Y.work = take(2 * sizeof(int32_t));  // the split-KV kernel's work counter and CTAs done
  Y.part_ml = take(sizeof(float2) * items * nq);
  Y.part_o = take(sizeof(float) * items * nq * d);
  Y.total = o;
  return Y;
}

// The loop's fixed metadata: one row per lane (row l = lane l = block l =
// readout l), the combine entries, and the RoPE frequencies base^(-2i/d)
// (double, rounded once to float).
__global__ void loop_init_kernel(DevMeta m, int L, int Hkv, int MC, int nq, int d, float base) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i == 0) {  // the persistent split-KV grid's counter starts from zero
    m.dec_work[0] = 0;
    m.dec_work[1] = 0;
  }
  if (i <= L) {
    const_cast<int32_t*>(m.row_indptr)[i] = i;
    const_cast<int32_t*>(m.ro_indptr)[i] = i;
  }
  if (i < L) {
    const_cast<int32_t*>(m.row_lane)[i] = i;
    const_cast<int32_t*>(m.readout)[i] = i;
    const_cast<int32_t*>(m.ro_idx)[i] = i;
    const_cast<int32_t*>(m.row_block)[i] = i;
    const_cast<int32_t*>(m.fold_count)[i] = 0;
  }
  if (i < L * Hkv)
    const_cast<CombEntry*>(m.comb)[i] = CombEntry{i * MC * nq, MC, nq, i / Hkv, -1, 0, 0, 0};
  if (i < d / 2)
    const_cast<float*>(m.rope_freq)[i] =
        static_cast<float>(pow(static_cast<double>(base), -2.0 * i / d));
}

// Step geometry from frozen_len, and the split-KV items over each lane's
// visible slots [0, kv_len) in kLoopChunk-slot chunks (chunks past kv_len are
// empty items, whose partial state is (-inf, 0)).
__global__ void loop_step_kernel(DevMeta m, int L, int Hkv, int MC, int nq, int P,
                                 const int32_t* frozen_len, int fold_mode, uint32_t* status) {
  grid_dep_wait();  // the previous step's fold
  grid_dep_launch();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < L * Hkv * MC) {
    const int c = i % MC, lg = i / MC, g = lg % Hkv, l = lg / Hkv;
    const int f = frozen_len[l];
    const int cap = (m.page_indptr[l + 1] - m.page_indptr[l]) * P;
    const bool ok = f >= 0 && f < cap;
    const int ext = ok ? f + 1 : 0;
    const int kb = c * kLoopChunk;
    const int ke = max(kb, min(ext, kb + kLoopChunk));
    const_cast<DecItem*>(m.dec_items)[i] = DecItem{l, g, l, 1, kb, ke, i * nq, -1};  // no list
    if (g == 0 && c == 0) {
      const_cast<int32_t*>(m.positions)[l] = f;
      const_cast<int32_t*>(m.slots)[l] = ok ? f : -1;  // -1: no slot, nothing is written
      const_cast<int32_t*>(m.kv_len)[l] = ext;
      const_cast<int32_t*>(m.fold_mode)[l] = ok ? fold_mode : PIE_FOLD_NONE;
      if (!ok) set_status(status, PIE_STATUS_LOOP_FULL);
    }
  }
}

}  // namespace pie

using namespace pie;

static int loop_check(const pie_fwd_desc* desc, int32_t num_lanes, int32_t max_pages, int& G,
                      int& nq, int& MC) {
  if (!desc) return set_last_error(PIE_EINVAL, "desc is NULL");
  const pie_fwd_desc& D = *desc;
  if (D.num_q_heads <= 0 || D.num_kv_heads <= 0 || D.num_q_heads % D.num_kv_heads != 0)
    return set_last_error(PIE_EINVAL, "num_q_heads must be a positive multiple of num_kv_heads");
  if ((D.head_dim != 64 && D.head_dim != 128) ||
      (D.page_size != 8 && D.page_size != 16 && D.page_size != 32) ||
      (D.dtype != PIE_F32 && D.dtype != PIE_BF16))
    return set_last_error(PIE_EUNSUPPORTED, "head_dim 64/128, page_size 8/16/32, f32/bf16 only");
  if (!(D.rope_base > 0.0f)) return set_last_error(PIE_EINVAL, "rope_base must be positive");
  G = D.num_q_heads / D.num_kv_heads;
  if (G > 8) return set_last_error(PIE_EUNSUPPORTED, "more than 8 q heads per kv head is not built");
  if (num_lanes < 0 || max_pages < 0) return set_last_error(PIE_EINVAL, "negative size");
  nq = G <= 2 ? 2 : (G <= 4 ? 4 : 8);
  const int64_t cap = static_cast<int64_t>(max_pages) * D.page_size;
  if (cap > (int64_t(1) << 30)) return set_last_error(PIE_ERANGE, "max_pages_per_lane too large");
  MC = cap > 0 ? static_cast<int>((cap + kLoopChunk - 1) / kLoopChunk) : 1;
  return PIE_OK;
}

extern "C" int pie_fwd_decode_loop_workspace_bytes(const pie_fwd_desc* desc, int32_t num_lanes,
                                                   int32_t max_pages_per_lane, size_t* bytes) {
  if (!bytes) return set_last_error(PIE_EINVAL, "bytes is NULL");
  int G = 0, nq = 0, MC = 0;
  const int rc = loop_check(desc, num_lanes, max_pages_per_lane, G, nq, MC);
  if (rc != PIE_OK) return rc;
  *bytes = loop_layout(num_lanes, desc->num_kv_heads, MC, nq, desc->head_dim).total;
  return PIE_OK;
}

extern "C" int pie_fwd_decode_loop(const pie_fwd_desc* desc, int32_t num_lanes, int32_t steps,
                                   const int32_t* page_indptr, const int32_t* page_ids,
                                   int32_t num_pool_pages, int32_t max_pages_per_lane,
                                   int32_t* frozen_len,
                                   const void* q, const void* k, const void* v, void* q_rot,
                                   void* k_pool, void* v_pool, void* out, float* lse,
                                   const int32_t* channel, void* workspace, size_t ws_bytes,
                                   uint32_t* status, void* stream) {
  int G = 0, nq = 0, MC = 0;
  int rc = loop_check(desc, num_lanes, max_pages_per_lane, G, nq, MC);
  if (rc != PIE_OK) return rc;
  if (steps < 0 || num_pool_pages < 0) return set_last_error(PIE_EINVAL, "negative size");
  if (num_lanes == 0 || steps == 0) return PIE_OK;
  if (!page_indptr || !page_ids || !frozen_len || !q || !k || !v || !q_rot || !k_pool ||
      !v_pool || !out)
    return set_last_error(PIE_EINVAL, "decode loop: a required pointer is NULL");
  const pie_fwd_desc& D = *desc;
  const int L = num_lanes, Hq = D.num_q_heads, Hkv = D.num_kv_heads, d = D.head_dim;
  const LoopLayout Y = loop_layout(L, Hkv, MC, nq, d);
  if (!workspace || ws_bytes < Y.total)
    return set_last_error(PIE_ENOSPACE, "workspace smaller than pie_fwd_decode_loop_workspace_bytes()");
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return set_last_error(PIE_EINVAL, "workspace must be 256-byte aligned");

  char* w = static_cast<char*>(workspace);
  pie_fwd_plan_t p;
  std::memset(&p, 0, sizeof(p));
  p.device_tables = true;  // the loop's set-up kernel writes them
  p.desc = D;
  if (p.desc.sm_scale == 0.0f) p.desc.sm_scale = 1.0f / sqrtf(static_cast<float>(d));
  p.L = L;
  p.N = L;
  p.R = L;
  p.G = G;
  p.nq = nq;
  p.tc_nt = 1;
  p.num_dec_items = L * Hkv * MC;
  p.num_part_slots = static_cast<int64_t>(L) * Hkv * MC * nq;
  p.num_comb_merge = L * Hkv;
  DevMeta& m = p.dev;
  m.row_indptr = reinterpret_cast<const int32_t*>(w + Y.row_indptr);
  m.row_lane = reinterpret_cast<const int32_t*>(w + Y.row_lane);
  m.positions = reinterpret_cast<const int32_t*>(w + Y.positions);
  m.slots = reinterpret_cast<const int32_t*>(w + Y.slots);
  m.kv_len = reinterpret_cast<const int32_t*>(w + Y.kv_len);
  m.fold_mode = reinterpret_cast<const int32_t*>(w + Y.fold_mode);
  m.fold_count = reinterpret_cast<const int32_t*>(w + Y.fold_count);
  m.readout = reinterpret_cast<const int32_t*>(w + Y.readout);
  m.ro_indptr = reinterpret_cast<const int32_t*>(w + Y.ro_indptr);
  m.ro_idx = reinterpret_cast<const int32_t*>(w + Y.ro_idx);
  m.rope_freq = reinterpret_cast<const float*>(w + Y.rope_freq);
  m.dec_items = reinterpret_cast<const DecItem*>(w + Y.dec);
  m.comb = reinterpret_cast<const CombEntry*>(w + Y.comb);
  m.row_block = reinterpret_cast<const int32_t*>(w + Y.row_block);
  m.part_ml = reinterpret_cast<float2*>(w + Y.part_ml);
  m.part_o = reinterpret_cast<float*>(w + Y.part_o);
  m.page_indptr = page_indptr;
  m.page_ids = page_ids;
  m.num_pool_pages = num_pool_pages;
  // each step's split-KV items go to a persistent grid sized for this device
  m.dec_work = reinterpret_cast<int32_t*>(w + Y.work);
  m.num_sms = device_sm_count();

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int init_n = std::max(L * Hkv, std::max(L + 1, d / 2));
  loop_init_kernel<<<(init_n + 255) / 256, 256, 0, s>>>(m, L, Hkv, MC, nq, d, D.rope_base);
  cudaError_t e = cudaGetLastError();
  const size_t esz = D.dtype == PIE_BF16 ? 2 : 4;
  const size_t q_step = static_cast<size_t>(L) * Hq * d * esz;
  const size_t kv_step = static_cast<size_t>(L) * Hkv * d * esz;
  const int items = L * Hkv * MC;
  for (int t = 0; t < steps && e == cudaSuccess; ++t) {
    e = launch_dependent(loop_step_kernel, dim3((items + 255) / 256), dim3(256), 0, s, true, m, L,
                         Hkv, MC, nq, D.page_size, frozen_len,
                         channel ? PIE_FOLD_CHANNEL : PIE_FOLD_ALL, status);
    if (e == cudaSuccess)
      e = launch_rope_scatter(p, static_cast<const char*>(q) + t * q_step,
                              static_cast<const char*>(k) + t * kv_step,
                              static_cast<const char*>(v) + t * kv_step, q_rot, k_pool, v_pool,
                              frozen_len, status, s);
    if (e == cudaSuccess)
      e = launch_attend_decode(p, q_rot, k_pool, v_pool, nullptr, status, s);
    if (e == cudaSuccess)
      e = launch_combine(p, static_cast<char*>(out) + t * q_step, lse ? lse + size_t(t) * L * Hq : nullptr,
                         nullptr, nullptr, s);
    if (e == cudaSuccess)
      e = launch_fold(p, frozen_len, channel ? channel + size_t(t) * L : nullptr, status, s);
  }
  if (e != cudaSuccess)
    return set_last_error(PIE_ECUDA, std::string("decode loop launch: ") + cudaGetErrorString(e));
  return PIE_OK;
}
