// CPU oracle for the data-parallel hot path of one Pie ForwardPass attention
// layer over a paged KV working set.
//
// TEST INFRASTRUCTURE ONLY.  The test-suite, the package smoke check and the
// benchmark's CPU-baseline leg are the only callers.  Nothing here is shared
// with the CUDA library: no header, helper, table or constant.  The library
// must never load this file.
//
// What it computes, in the plain order of the definitions (Pie, "The forward
// pass": Lanes; State geometry table; Attention masks; Readouts):
//   1. validate the pass metadata (lanes by row indptr; StateGeometry fields
//      positions/slots per row, kv_len/fold per lane; working sets as page
//      lists; a row's writes must not collide, Pie review Eq. (4));
//   2. rotate q and k of every row at its explicit position (RoPE) and write
//      the row's K/V into its slot of its lane's working set, through the
//      page table;
//   3. attention of every row and query head over the lane's first kv_len
//      slots, restricted to the row's visible set (default causal in slot
//      space, or the row's bitmask), accumulated in double precision;
//   4. gather the readout rows (default: last row of every lane);
//   5. fold: freeze none / all / a count / a count read from a channel of
//      the lane's newly written slots.
// Pool layout: [num_pages][num_kv_heads][page_size][head_dim].
//
// Readings where the pages leave a step open (each is also listed in the
// design notes): rotate-half RoPE with an fp32 angle; default visibility =
// slot <= own slot and < kv_len; a mask replaces the default and is
// intersected with kv_len; an empty visible set gives o = 0, lse = -inf;
// softmax scale 1/sqrt(d); q head h reads kv head h / (Hq/Hkv); a fold
// freezes the first k new slots (which must follow the frozen prefix);
// channel counts outside [0, n] are clamped and flagged.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

extern "C" {

// ---- own error codes and status bits -------------------------------------
enum {
  ORC_OK = 0,
  ORC_EINVAL = -1,   // malformed metadata
  ORC_ERANGE = -2,   // a value outside its allowed range
};
enum {
  ORC_ST_FROZEN_WRITE = 1u,  // a row targeted a frozen slot; write skipped
  ORC_ST_FOLD_CLAMP = 2u,    // a channel fold count was clamped to [0, n]
  ORC_ST_FOLD_GAP = 8u,      // a folding lane's first slot != frozen length
};
enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_FOLD_NONE = 0, ORC_FOLD_ALL = 1, ORC_FOLD_COUNT = 2, ORC_FOLD_CHANNEL = 3 };

typedef struct {
  int32_t num_q_heads, num_kv_heads, head_dim, page_size, dtype;
  double rope_base;
  double sm_scale;  // 0 => 1/sqrt(head_dim)
} orc_desc;

typedef struct {
  int32_t num_lanes, num_rows;
  const int32_t* row_indptr;    // [L+1]
  const int32_t* positions;     // [N]
  const int32_t* slots;         // [N]
  const int32_t* kv_len;        // [L]
  const int32_t* page_indptr;   // [L+1]
  const int32_t* page_ids;      // [page_indptr[L]]
  int32_t num_pool_pages;
  const int32_t* fold_mode;     // [L]
  const int32_t* fold_count;    // [L]
  const int64_t* mask_word_indptr;  // [N+1] or NULL (default visibility)
  const int32_t* readout;       // [R] or NULL (last row of every lane)
  int32_t num_readout;
} orc_meta;

}  // extern "C"

namespace {

// ---- dtype storage ---------------------------------------------------------
double bf16_to_double(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

// Round a double to the nearest bfloat16 (ties to even), directly from the
// double (no intermediate float rounding).
uint16_t double_to_bf16(double x) {
  if (std::isnan(x)) return 0x7FC0;
  uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  double a = std::fabs(x);
  if (a == 0.0) return sign;
  int e;
  std::frexp(a, &e);  // a = m * 2^e, m in [0.5, 1)
  // bf16: 8 significant bits for normals (exponent >= -125 in frexp terms),
  // subnormal quantum 2^-133.
  int q_exp = (e - 1 >= -126) ? (e - 8) : (-133);
  double quantum = std::ldexp(1.0, q_exp);
  double n = std::nearbyint(a / quantum);  // exact division by a power of two
  double r = n * quantum;
  const double max_bf16 = std::ldexp(255.0, 120);  // (2 - 2^-7) * 2^127
  if (r > max_bf16) return sign | 0x7F80;         // overflow to infinity
  float f = static_cast<float>(r);                // exact: r has <= 8 bits
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return sign | static_cast<uint16_t>((u >> 16) & 0x7FFF);
}

double load(int dtype, const void* p, size_t i) {
  if (dtype == ORC_F32) return static_cast<double>(static_cast<const float*>(p)[i]);
  return bf16_to_double(static_cast<const uint16_t*>(p)[i]);
}

void store(int dtype, void* p, size_t i, double x) {
  if (dtype == ORC_F32)
    static_cast<float*>(p)[i] = static_cast<float>(x);
  else
    static_cast<uint16_t*>(p)[i] = double_to_bf16(x);
}

// ---- RoPE (rotate-half pairing of i and i + d/2) ----------------------------
// Frequency of pair i: base^(-2i/d), computed in double and rounded once to
// float; angle = float(pos) * freq as one float multiply; cos/sin evaluated
// in double on that float angle.  The rotated pair is
//   x'[i]       = x[i] cos - x[i + d/2] sin
//   x'[i + d/2] = x[i + d/2] cos + x[i] sin.
void rope(const orc_desc& D, const double* x, int32_t pos, double* out) {
  const int d = D.head_dim, h = d / 2;
  for (int i = 0; i < h; ++i) {
    float freq = static_cast<float>(std::pow(D.rope_base, -2.0 * i / d));
    float theta = static_cast<float>(pos) * freq;
    double c = std::cos(static_cast<double>(theta));
    double s = std::sin(static_cast<double>(theta));
    out[i] = x[i] * c - x[i + h] * s;
    out[i + h] = x[i + h] * c + x[i] * s;
  }
}

int lane_rows(const orc_meta& M, int l) { return M.row_indptr[l + 1] - M.row_indptr[l]; }

bool mask_bit(const uint32_t* words, int64_t base, int s) {
  return (words[base + (s >> 5)] >> (s & 31)) & 1u;
}

}  // namespace

extern "C" {

// Physical element offset of (slot s of lane l, kv head g, dim 0) in a pool.
static size_t pool_offset(const orc_desc& D, const orc_meta& M, int l, int s, int g) {
  int page = M.page_ids[M.page_indptr[l] + s / D.page_size];
  return ((static_cast<size_t>(page) * D.num_kv_heads + g) * D.page_size + s % D.page_size) *
         D.head_dim;
}

// Step 1: metadata checks.  Returns ORC_OK or an error code; nothing is
// written.
int orc_validate(const orc_desc* desc, const orc_meta* meta) {
  const orc_desc& D = *desc;
  const orc_meta& M = *meta;
  if (D.num_q_heads <= 0 || D.num_kv_heads <= 0 || D.head_dim <= 0 || D.page_size <= 0)
    return ORC_EINVAL;
  if (D.num_q_heads % D.num_kv_heads != 0 || D.head_dim % 2 != 0) return ORC_EINVAL;
  if (D.dtype != ORC_F32 && D.dtype != ORC_BF16) return ORC_EINVAL;
  if (M.num_lanes < 0 || M.num_rows < 0 || M.num_pool_pages < 0) return ORC_EINVAL;
  if (!M.row_indptr || !M.kv_len || !M.page_indptr || !M.fold_mode) return ORC_EINVAL;
  if (M.num_rows > 0 && (!M.positions || !M.slots)) return ORC_EINVAL;
  if (M.row_indptr[0] != 0 || M.row_indptr[M.num_lanes] != M.num_rows) return ORC_EINVAL;
  if (M.page_indptr[0] != 0) return ORC_EINVAL;
  for (int l = 0; l < M.num_lanes; ++l) {
    if (M.row_indptr[l + 1] < M.row_indptr[l]) return ORC_EINVAL;
    if (M.page_indptr[l + 1] < M.page_indptr[l]) return ORC_EINVAL;
  }
  if (M.page_indptr[M.num_lanes] > 0 && !M.page_ids) return ORC_EINVAL;
  for (int64_t i = 0; i < M.page_indptr[M.num_lanes]; ++i)
    if (M.page_ids[i] < 0 || M.page_ids[i] >= M.num_pool_pages) return ORC_ERANGE;
  for (int l = 0; l < M.num_lanes; ++l) {
    const int64_t cap =
        static_cast<int64_t>(M.page_indptr[l + 1] - M.page_indptr[l]) * D.page_size;
    if (M.kv_len[l] < 0 || M.kv_len[l] > cap) return ORC_ERANGE;
    const int n = lane_rows(M, l);
    for (int r = M.row_indptr[l]; r < M.row_indptr[l + 1]; ++r) {
      if (M.positions[r] < 0) return ORC_ERANGE;
      if (M.slots[r] < 0 || M.slots[r] >= cap) return ORC_ERANGE;
    }
    const int fm = M.fold_mode[l];
    if (fm < ORC_FOLD_NONE || fm > ORC_FOLD_CHANNEL) return ORC_EINVAL;
    if (fm == ORC_FOLD_COUNT) {
      if (!M.fold_count) return ORC_EINVAL;
      if (M.fold_count[l] < 0 || M.fold_count[l] > n) return ORC_ERANGE;
    }
    if (fm != ORC_FOLD_NONE) {
      // a fold freezes the first k new slots, so they must be consecutive
      for (int r = M.row_indptr[l] + 1; r < M.row_indptr[l + 1]; ++r)
        if (M.slots[r] != M.slots[r - 1] + 1) return ORC_EINVAL;
    }
  }
  // Eq. (4): no two rows of the pass may write the same physical slot.
  {
    std::vector<int64_t> t;
    t.reserve(M.num_rows);
    for (int l = 0; l < M.num_lanes; ++l)
      for (int r = M.row_indptr[l]; r < M.row_indptr[l + 1]; ++r) {
        int s = M.slots[r];
        int64_t page = M.page_ids[M.page_indptr[l] + s / D.page_size];
        t.push_back(page * D.page_size + s % D.page_size);
      }
    // sort the physical targets and look for equal neighbours
    std::sort(t.begin(), t.end());
    for (size_t i = 1; i < t.size(); ++i)
      if (t[i] == t[i - 1]) return ORC_EINVAL;
  }
  if (M.mask_word_indptr) {
    if (M.mask_word_indptr[0] != 0) return ORC_EINVAL;
    for (int l = 0; l < M.num_lanes; ++l)
      for (int r = M.row_indptr[l]; r < M.row_indptr[l + 1]; ++r) {
        int64_t nw = M.mask_word_indptr[r + 1] - M.mask_word_indptr[r];
        if (nw < 0) return ORC_EINVAL;
        if (nw < (static_cast<int64_t>(M.kv_len[l]) + 31) / 32) return ORC_ERANGE;
      }
  }
  if (M.readout) {
    if (M.num_readout < 0) return ORC_EINVAL;
    for (int j = 0; j < M.num_readout; ++j)
      if (M.readout[j] < 0 || M.readout[j] >= M.num_rows) return ORC_ERANGE;
  }
  return ORC_OK;
}

// Step 2: RoPE + slot scatter.  q_rot [N,Hq,d] is written in the dtype;
// k_pool/v_pool are updated in place.  A row whose slot lies in the lane's
// frozen prefix is not written and sets ORC_ST_FROZEN_WRITE.  A lane that
// will fold but whose first new slot is not its frozen length sets
// ORC_ST_FOLD_GAP.  Rows are applied in row order.
void orc_append_kv(const orc_desc* desc, const orc_meta* meta, const void* q, const void* k,
                   const void* v, void* q_rot, void* k_pool, void* v_pool,
                   const int32_t* frozen_len, uint32_t* status) {
  const orc_desc& D = *desc;
  const orc_meta& M = *meta;
  const int d = D.head_dim, Hq = D.num_q_heads, Hkv = D.num_kv_heads;
  std::vector<double> x(d), y(d);
  for (int l = 0; l < M.num_lanes; ++l) {
    if (M.fold_mode[l] != ORC_FOLD_NONE && lane_rows(M, l) > 0 &&
        M.slots[M.row_indptr[l]] != frozen_len[l])
      *status |= ORC_ST_FOLD_GAP;
    for (int r = M.row_indptr[l]; r < M.row_indptr[l + 1]; ++r) {
      const int pos = M.positions[r];
      for (int h = 0; h < Hq; ++h) {
        size_t base = (static_cast<size_t>(r) * Hq + h) * d;
        for (int j = 0; j < d; ++j) x[j] = load(D.dtype, q, base + j);
        rope(D, x.data(), pos, y.data());
        for (int j = 0; j < d; ++j) store(D.dtype, q_rot, base + j, y[j]);
      }
      const int s = M.slots[r];
      if (s < frozen_len[l]) {
        *status |= ORC_ST_FROZEN_WRITE;
        continue;
      }
      for (int g = 0; g < Hkv; ++g) {
        size_t src = (static_cast<size_t>(r) * Hkv + g) * d;
        size_t dst = pool_offset(D, M, l, s, g);
        for (int j = 0; j < d; ++j) x[j] = load(D.dtype, k, src + j);
        rope(D, x.data(), pos, y.data());
        for (int j = 0; j < d; ++j) store(D.dtype, k_pool, dst + j, y[j]);
        // v is not rotated: copied bit for bit
        const size_t eb = D.dtype == ORC_F32 ? 4 : 2;
        std::memcpy(static_cast<char*>(v_pool) + dst * eb,
                    static_cast<const char*>(v) + src * eb, d * eb);
      }
    }
  }
}

// Visible-set predicate of row r (lane l) for slot s (step 3's V(r)).
static bool visible(const orc_meta& M, const uint32_t* mask_words, int l, int r, int s) {
  if (s >= M.kv_len[l]) return false;
  if (M.mask_word_indptr && mask_words) return mask_bit(mask_words, M.mask_word_indptr[r], s);
  return s <= M.slots[r];
}

// Step 3: attention.  For every row r in `rows` (NULL => all rows) and every
// query head h:  z_s = scale * <q_rot[r,h], K[s, h/G]> over visible slots s in
// ascending order, m = max z, o = sum e^(z_s - m) V[s] / sum e^(z_s - m),
// lse = m + ln(sum e^(z_s - m)).  Empty visible set => o = 0, lse = -inf.
// out [N,Hq,d] and lse [N,Hq] are double.  The pools are only read.
void orc_attend(const orc_desc* desc, const orc_meta* meta, const void* q_rot,
                const void* k_pool, const void* v_pool, const uint32_t* mask_words,
                const int32_t* rows, int32_t num_sel, double* out, double* lse,
                int32_t num_threads) {
  const orc_desc& D = *desc;
  const orc_meta& M = *meta;
  const int d = D.head_dim, Hq = D.num_q_heads, Hkv = D.num_kv_heads;
  const int G = Hq / Hkv;
  const double scale = D.sm_scale != 0.0 ? D.sm_scale : 1.0 / std::sqrt(static_cast<double>(d));
  std::vector<int> row_lane(M.num_rows);
  for (int l = 0; l < M.num_lanes; ++l)
    for (int r = M.row_indptr[l]; r < M.row_indptr[l + 1]; ++r) row_lane[r] = l;
  std::vector<int> todo;
  if (rows) {
    todo.assign(rows, rows + num_sel);
  } else {
    for (int r = 0; r < M.num_rows; ++r) todo.push_back(r);
  }
  auto work = [&](size_t lo, size_t hi) {
    std::vector<double> qv(d), z, acc(d);
    std::vector<int> vis;
    for (size_t t = lo; t < hi; ++t) {
      const int r = todo[t], l = row_lane[r];
      vis.clear();
      for (int s = 0; s < M.kv_len[l]; ++s)
        if (visible(M, mask_words, l, r, s)) vis.push_back(s);
      for (int h = 0; h < Hq; ++h) {
        const int g = h / G;
        double* o = out + (static_cast<size_t>(r) * Hq + h) * d;
        double& L = lse[static_cast<size_t>(r) * Hq + h];
        if (vis.empty()) {
          for (int j = 0; j < d; ++j) o[j] = 0.0;
          L = -std::numeric_limits<double>::infinity();
          continue;
        }
        size_t qb = (static_cast<size_t>(r) * Hq + h) * d;
        for (int j = 0; j < d; ++j) qv[j] = load(D.dtype, q_rot, qb + j);
        z.assign(vis.size(), 0.0);
        double m = -std::numeric_limits<double>::infinity();
        for (size_t i = 0; i < vis.size(); ++i) {
          size_t kb = pool_offset(D, M, l, vis[i], g);
          double dot = 0.0;
          for (int j = 0; j < d; ++j) dot += qv[j] * load(D.dtype, k_pool, kb + j);
          z[i] = scale * dot;
          if (z[i] > m) m = z[i];
        }
        double sum = 0.0;
        std::fill(acc.begin(), acc.end(), 0.0);
        for (size_t i = 0; i < vis.size(); ++i) {
          double w = std::exp(z[i] - m);
          sum += w;
          size_t vb = pool_offset(D, M, l, vis[i], g);
          for (int j = 0; j < d; ++j) acc[j] += w * load(D.dtype, v_pool, vb + j);
        }
        for (int j = 0; j < d; ++j) o[j] = acc[j] / sum;
        L = m + std::log(sum);
      }
    }
  };
  int T = num_threads > 1 ? num_threads : 1;
  if (T == 1 || todo.size() < 2) {
    work(0, todo.size());
    return;
  }
  std::vector<std::thread> th;
  size_t per = (todo.size() + T - 1) / T;
  for (int i = 0; i < T; ++i) {
    size_t lo = i * per, hi = std::min(todo.size(), lo + per);
    if (lo >= hi) break;
    th.emplace_back(work, lo, hi);
  }
  for (auto& t : th) t.join();
}

// Step 4: the readout rows.  Writes up to `cap` row indices and returns R
// (the given list, else the last row of every lane that has rows).
int32_t orc_readout_rows(const orc_meta* meta, int32_t* out, int32_t cap) {
  const orc_meta& M = *meta;
  int32_t R = 0;
  if (M.readout) {
    for (int j = 0; j < M.num_readout; ++j) {
      if (R < cap) out[R] = M.readout[j];
      ++R;
    }
    return R;
  }
  for (int l = 0; l < M.num_lanes; ++l)
    if (lane_rows(M, l) > 0) {
      if (R < cap) out[R] = M.row_indptr[l + 1] - 1;
      ++R;
    }
  return R;
}

// Step 5: fold.  k = 0 (none), n (all), fold_count (literal) or the channel
// value clamped to [0, n] (ORC_ST_FOLD_CLAMP when clamped); frozen_len += k.
void orc_fold(const orc_meta* meta, int32_t* frozen_len, const int32_t* channel,
              uint32_t* status) {
  const orc_meta& M = *meta;
  for (int l = 0; l < M.num_lanes; ++l) {
    const int n = lane_rows(M, l);
    int k = 0;
    switch (M.fold_mode[l]) {
      case ORC_FOLD_NONE: k = 0; break;
      case ORC_FOLD_ALL: k = n; break;
      case ORC_FOLD_COUNT: k = M.fold_count[l]; break;
      case ORC_FOLD_CHANNEL: {
        int c = channel[l];
        k = c < 0 ? 0 : (c > n ? n : c);
        if (k != c) *status |= ORC_ST_FOLD_CLAMP;
        break;
      }
    }
    frozen_len[l] += k;
  }
}

// Eq. (1) of the Pie review: bytes of a dense K+V cache.
int64_t orc_kv_bytes(int64_t layers, int64_t kv_heads, int64_t head_dim, int64_t tokens,
                     int64_t elem_bytes) {
  return 2 * layers * kv_heads * head_dim * tokens * elem_bytes;
}

// Eq. (2) of the Pie review: unused slots in the last page.
int64_t orc_page_waste(int64_t tokens, int64_t page_size) {
  return page_size * ((tokens + page_size - 1) / page_size) - tokens;
}

// Exposed for pins: the rounding the oracle applies when storing bf16.
uint16_t orc_round_bf16(double x) { return double_to_bf16(x); }

// Exposed for pins: RoPE of one head vector (double in, double out).
void orc_rope(const orc_desc* desc, const double* x, int32_t pos, double* out) {
  rope(*desc, x, pos, out);
}

}  // extern "C"
