// Readout distribution epilogue: the top-K candidates of the next-token
// distribution of every readout row (the review "Pie: Who Should Control the
// LLM Generation Loop?", section 7, Eq. (6)-(7): the serving system returns
// the K = 256 most probable tokens of a ~128K-token distribution, their
// probabilities and the mass Z they keep; 1 - Z is the total-variation
// distance of Eq. (7) when a client renormalises them).
//
// p = softmax(logits row); the k tokens of largest p, ties by smaller token
// id; their p (not renormalised), Z = the sum of those p, and the natural-log
// normaliser lse.  The pass is bound by HBM (the logits are read once, ~0.5 MB
// per row at 128K fp32 tokens), so a row is cut into parts read by many CTAs:
//   1. filter kernel, grid (rows, parts), 512 threads: a 16,384-token part
//      into registers (32 tokens per thread, coalesced 16-byte loads), the
//      part's max and sum of exp(x - max), and a short unsorted list of
//      (key, token) candidates: every token at or above a lower bound on the
//      part's k-th largest logit.  The bound is the k-th largest of the 512
//      thread maxima (k distinct tokens reach it), found to within 1/4,096 of
//      their range by one shared-memory histogram whose bins span exactly
//      [min, max] of those maxima; about 2 % of a part is listed.  A part
//      whose list would pass 512 entries (ties, flat rows) sets a flag;
//   2. slice kernel, grid (rows, slices), 512 threads, only for flagged rows:
//      a 8,192-token slice into shared memory as order-preserving 32-bit keys,
//      its max and sum, then its exact k largest (a 4,096-bin histogram of the
//      top 12 key bits finds the bucket of the k-th key; the keys in it or
//      above are listed in token order and an exact radix select over the
//      list, or over the whole slice when ties crowd the bucket, yields k
//      (key, token) candidates);
//   3. merge kernel, one CTA per row: over the row's candidates (the parts'
//      lists, or the slices' k each), an exact radix select of the k-th
//      largest key (12-, 10- and 10-bit passes) and, when that key has more
//      copies than places, of the smallest tokens among them (two 10-bit
//      passes); a bitonic sort of the k as 64-bit (key, ~token) words; the
//      (max, sum) pairs merge into lse, and p = exp(x - lse) and Z follow.
// Every token the row can return is a candidate: each part lists all of its
// tokens at or above a bound that is at most the row's k-th largest logit,
// and the row's top k lie in the union of its slices' top k.

#include <cmath>
#include <string>

#include "common.cuh"

namespace pie {

namespace ro {

constexpr int kSlice = 8192;            // tokens per slice
constexpr int kThreads = 512;
constexpr int kPer = kSlice / kThreads;  // tokens per thread (a contiguous run)
constexpr int kMaxK = 256;
constexpr int kMaxSlices = 32;           // vocab <= 262,144: the merge takes <= 8,192 candidates
constexpr int kMergeThreads = 1024;
constexpr int kListCap = 1024;           // keys the slice kernel's exact selection takes from a list
constexpr int kPart = 16384;             // tokens per part of the filter kernel
constexpr int kFThreads = 512;
constexpr int kFPer = kPart / kFThreads; // tokens per thread, in registers
constexpr int kFCap = 512;               // candidates a part may list (more: the row takes the slices)
constexpr int kMaxParts = 16;            // vocab <= 262,144
constexpr int kWin = 4096;               // bins of the thread-maxima histogram
static_assert(kMaxParts * kFCap == kMaxSlices * kMaxK, "the merge holds either candidate set");

// Shared-memory position of slice token i: one pad word every 32 words, so
// that thread t reading token t * 32 + c (its run) hits bank (t + c) % 32.
__device__ __forceinline__ int spos(int i) { return i + (i >> 5); }

// Order-preserving key of a float (larger float, larger key); -0 counts as +0.
__device__ __forceinline__ uint32_t key_of(float x) {
  uint32_t b = __float_as_uint(x);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float value_of(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Exclusive prefix over the NT threads of v; *total gets the block total.
template <int NT>
__device__ __forceinline__ int block_scan(int v, int* warp_sums, int* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += u;
  }
  __syncthreads();
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < NT / 32 ? warp_sums[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += u;
    }
    if (lane < NT / 32) warp_sums[lane] = wi - w;
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  return warp_sums[warp] + incl - v;
}

struct SelectSmem {
  int hist[4096];
  int warp_sums[32];
  int total, bin, above, bin_cnt;
};

// After a histogram of nbins bins: the bin holding the rem-th largest value,
// bins taken from the top -> sm.bin, the count in the bins above it ->
// sm.above, its own count -> sm.bin_cnt.  Thread t takes nbins / NT
// consecutive bins from the top; a block scan of their counts finds the bin.
template <int NT>
__device__ void pick_bin(int nbins, int rem, SelectSmem& sm) {
  const int t = threadIdx.x;
  const int per = nbins / NT;
  const int top = nbins - 1 - t * per;
  int cnt = 0;
  for (int q = 0; q < per; ++q) cnt += sm.hist[top - q];
  const int excl = block_scan<NT>(cnt, sm.warp_sums, &sm.total);
  if (excl < rem && rem <= excl + cnt) {
    int acc = excl;
    for (int q = 0; q < per; ++q) {
      const int c = sm.hist[top - q];
      if (acc + c >= rem) {
        sm.bin = top - q;
        sm.above = acc;
        sm.bin_cnt = c;
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

// The kk-th largest of the block's keys (E per thread, held in registers;
// key 0 is padding, below every token): a radix select on bits 31..20 (4,096
// bins: the sign, the exponent and three mantissa bits, so a block's keys
// spread over many bins and the shared-memory adds rarely collide), then
// 19..10 and 9..0 among the keys sharing the prefix chosen so far.  Returns
// the key; need_eq = how many keys equal to it belong to the kk (the others
// are the keys above it); sm.bin_cnt is left holding how many keys equal it.
template <int NT, int E>
__device__ uint32_t select_kth(const uint32_t (&key)[E], int kk, SelectSmem& sm, int& need_eq) {
  const int t = threadIdx.x;
  uint32_t prefix = 0u, pmask = 0u;
  int rem = kk;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 20 : (pass == 1 ? 10 : 0);
    const int nbins = pass == 0 ? 4096 : 1024;
    const uint32_t bmask = uint32_t(nbins - 1);
    for (int i = t; i < nbins; i += NT) sm.hist[i] = 0;
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (key[e] != 0u && (key[e] & pmask) == prefix)
        atomicAdd(&sm.hist[(key[e] >> shift) & bmask], 1);
    __syncthreads();
    pick_bin<NT>(nbins, rem, sm);
    rem -= sm.above;
    prefix |= uint32_t(sm.bin) << shift;
    pmask |= bmask << shift;
    __syncthreads();  // hist, bin and above are rewritten by the next pass
  }
  need_eq = rem;
  return prefix;
}

// Tokens below 2^20 ranked smallest first: a larger rank, a smaller token.
constexpr uint32_t kTokRank = (1u << 20) - 1u;

// Among the keys equal to thr (tokens distinct), the rank (kTokRank - token)
// of the rem-th smallest token: a radix select of the rank on bits 19..10,
// then 9..0.  The keys equal to thr with a rank at or above the result are
// the rem smallest tokens.
template <int NT, int E>
__device__ uint32_t select_tok(const uint32_t (&key)[E], const uint32_t (&tok)[E], uint32_t thr,
                               int rem, SelectSmem& sm) {
  const int t = threadIdx.x;
  uint32_t prefix = 0u, pmask = 0u;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 10 : 0;
    for (int i = t; i < 1024; i += NT) sm.hist[i] = 0;
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const uint32_t u = kTokRank - tok[e];
      if (key[e] != 0u && key[e] == thr && (u & pmask) == prefix)
        atomicAdd(&sm.hist[(u >> shift) & 1023u], 1);
    }
    __syncthreads();
    pick_bin<NT>(1024, rem, sm);
    rem -= sm.above;
    prefix |= uint32_t(sm.bin) << shift;
    pmask |= 1023u << shift;
    __syncthreads();
  }
  return prefix;
}

// From a complete 4,096-bin histogram of the top 12 key bits: the bin that
// holds the kk-th largest key, and how many keys lie in that bin or above it.
template <int NT>
__device__ uint32_t find_bucket(int kk, SelectSmem& sm, int& count_ge) {
  const int t = threadIdx.x;
  const int per = 4096 / NT;
  const int top = 4095 - t * per;
  int cnt = 0;
  for (int q = 0; q < per; ++q) cnt += sm.hist[top - q];
  const int excl = block_scan<NT>(cnt, sm.warp_sums, &sm.total);
  if (t == 0) {  // fewer than kk keys in all: every bin
    sm.bin = 0;
    sm.above = sm.total;
  }
  __syncthreads();
  if (excl < kk && kk <= excl + cnt) {
    int acc = excl;
    for (int q = 0; q < per; ++q) {
      const int c = sm.hist[top - q];
      if (acc + c >= kk) {
        sm.bin = top - q;
        sm.above = acc + c;
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
  count_ge = sm.above;
  const uint32_t b = uint32_t(sm.bin);
  __syncthreads();
  return b;
}

// The 4,096-bin coarse pass over the block's keys (E per thread, key 0 =
// padding) and its bucket.
template <int NT, int E>
__device__ uint32_t coarse_bin(const uint32_t (&key)[E], int kk, SelectSmem& sm, int& count_ge) {
  const int t = threadIdx.x;
  for (int i = t; i < 4096; i += NT) sm.hist[i] = 0;
  __syncthreads();
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (key[e] != 0u) atomicAdd(&sm.hist[key[e] >> 20], 1);
  __syncthreads();
  return find_bucket<NT>(kk, sm, count_ge);
}

// Token of a thread's e-th key: a run of consecutive tokens, or a list.
struct TokRun {
  uint32_t first;
  __device__ uint32_t operator()(int e) const { return first + uint32_t(e); }
};
template <int E>
struct TokList {
  const uint32_t (&tok)[E];
  __device__ uint32_t operator()(int e) const { return tok[e]; }
};

// The kk keys of select_kth, in the order they are held (thread-major):
// every key above thr, then the first need_eq keys equal to thr, ranked by a
// block scan -- with the keys in token order, ties go to the smaller tokens.
template <int NT, int E, typename Tok>
__device__ void emit_selected(const uint32_t (&key)[E], Tok tok, uint32_t thr, int need_eq,
                              SelectSmem& sm, uint2* out) {
  int my_gt = 0, my_eq = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    my_gt += key[e] > thr;
    my_eq += key[e] == thr;
  }
  int wg = block_scan<NT>(my_gt, sm.warp_sums, &sm.total);
  const int gt_total = sm.total;
  __syncthreads();
  int we = block_scan<NT>(my_eq, sm.warp_sums, &sm.total);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (key[e] > thr) {
      out[wg++] = make_uint2(key[e], tok(e));
    } else if (key[e] == thr) {
      if (we < need_eq) out[gt_total + we] = make_uint2(key[e], tok(e));
      ++we;
    }
  }
}

// Keys of the block (E per thread, in token order thread-major) at or above
// the coarse bucket cb, copied in that order to lkey / ltok.
template <int NT, int E, typename Tok>
__device__ void gather_list(const uint32_t (&key)[E], Tok tok, uint32_t cb, SelectSmem& sm,
                            uint32_t* lkey, uint32_t* ltok) {
  int mine = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) mine += key[e] != 0u && (key[e] >> 20) >= cb;
  int pos = block_scan<NT>(mine, sm.warp_sums, &sm.total);
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (key[e] != 0u && (key[e] >> 20) >= cb) {
      lkey[pos] = key[e];
      ltok[pos] = tok(e);
      ++pos;
    }
  __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 2) slice_kernel(const T* __restrict__ logits, int64_t ld,
                                                          int vocab, int k, int nslices,
                                                          uint2* __restrict__ cand,
                                                          float2* __restrict__ stats,
                                                          const int* __restrict__ ovf, int nparts) {
  extern __shared__ uint32_t keys[];  // spos(kSlice) words
  __shared__ SelectSmem sel;
  __shared__ float2 red2[kThreads / 32];
  __shared__ __align__(16) uint32_t lkey[kListCap];
  __shared__ uint32_t ltok[kListCap];
  const int r = blockIdx.x, s = blockIdx.y;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  // only rows whose parts overflowed their lists come here
  bool any = false;
  for (int p = 0; p < nparts; ++p) any = any || ovf[int64_t(r) * nparts + p] != 0;
  if (!any) return;
  const int base = s * kSlice;
  const int n = min(kSlice, vocab - base);
  const int kk = min(k, n);
  const T* row = logits + int64_t(r) * ld + base;

  // ---- load: coalesced 16-byte vectors, keys into shared memory (to be
  // re-read as each thread's contiguous run of tokens), the max and the sum
  constexpr int W = 16 / sizeof(T);
  {
    float v[kPer];
#pragma unroll
    for (int j = 0; j < kPer / W; ++j) {
      const int i0 = (j * kThreads + t) * W;
      float f[W];
      if (i0 + W <= n) {
        unpack16<T>(*reinterpret_cast<const uint4*>(row + i0), f);
      } else {
#pragma unroll
        for (int e = 0; e < W; ++e) f[e] = i0 + e < n ? Elem<T>::to_f(row[i0 + e]) : -INFINITY;
      }
#pragma unroll
      for (int e = 0; e < W; ++e) {
        v[j * W + e] = f[e];
        keys[spos(i0 + e)] = i0 + e < n ? key_of(f[e]) : 0u;  // padding below every token
      }
    }
    // (max, sum of exp(x - max)) of the thread's values, then merged across
    // the block in one reduction: (m1, s1) + (m2, s2) -> (m, s1 e^(m1-m) + s2 e^(m2-m))
    constexpr float kL2e = 1.4426950408889634f;
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPer; ++i) m = fmaxf(m, v[i]);
    float sum = 0.f;
    if (m != -INFINITY) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) sum += ex2((v[i] - m) * kL2e);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float mo = __shfl_xor_sync(0xffffffffu, m, off);
      const float so = __shfl_xor_sync(0xffffffffu, sum, off);
      const float mm = fmaxf(m, mo);
      sum = (m == -INFINITY ? 0.f : sum * ex2((m - mm) * kL2e)) +
            (mo == -INFINITY ? 0.f : so * ex2((mo - mm) * kL2e));
      m = mm;
    }
    if (lane == 0) red2[warp] = make_float2(m, sum);
    __syncthreads();
    if (t == 0) {
      float M = -INFINITY, S = 0.f;
      for (int w = 0; w < kThreads / 32; ++w) M = fmaxf(M, red2[w].x);
      for (int w = 0; w < kThreads / 32; ++w)
        if (red2[w].x != -INFINITY) S += red2[w].y * ex2((red2[w].x - M) * kL2e);
      stats[int64_t(r) * nslices + s] = make_float2(M, S);
    }
  }
  // ---- each thread's run of 32 consecutive tokens, in registers
  uint32_t key[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) key[i] = keys[spos(t * kPer + i)];
  uint2* out = cand + (int64_t(r) * nslices + s) * k;
  // ---- one coarse pass finds the 4,096-bin bucket of the kk-th key; the keys
  // in it or above (a few hundred for a peaked distribution) are copied, in
  // token order, to a short list, and the exact selection runs on the list
  int count_ge = 0;
  const uint32_t cb = coarse_bin<kThreads, kPer>(key, kk, sel, count_ge);
  if (count_ge <= kListCap) {
    gather_list<kThreads, kPer>(key, TokRun{uint32_t(base + t * kPer)}, cb, sel, lkey, ltok);
    constexpr int E2 = kListCap / kThreads;
    uint32_t lk[E2], lt[E2];
#pragma unroll
    for (int e = 0; e < E2; ++e) {
      const int i = t * E2 + e;
      lk[e] = i < count_ge ? lkey[i] : 0u;
      lt[e] = i < count_ge ? ltok[i] : 0u;
    }
    int need_eq = 0;
    const uint32_t thr = select_kth<kThreads, E2>(lk, kk, sel, need_eq);
    emit_selected<kThreads, E2>(lk, TokList<E2>{lt}, thr, need_eq, sel, out);
  } else {
    // ties or a flat distribution crowd the bucket: select over all keys
    int need_eq = 0;
    const uint32_t thr = select_kth<kThreads, kPer>(key, kk, sel, need_eq);
    emit_selected<kThreads, kPer>(key, TokRun{uint32_t(base + t * kPer)}, thr, need_eq, sel, out);
  }
}

// 64-bit words compared as the sort order: key, then smaller token first.
__device__ __forceinline__ unsigned long long sort_word(uint32_t key, uint32_t tok) {
  return (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - tok);
}

// Filter kernel, grid (rows, parts), 512 threads: one 16,384-token part of a
// row, 32 tokens per thread in registers, thread t holding tokens
// (j * 512 + t) * W + e (j < 32 / W, e < W; W tokens per 16-byte load).
//  - The thread's max and sum of exp(x - max), merged over the block: the
//    part's (max, sum) for the row's normaliser.
//  - The kk-th largest of the thread maxima (kk = min(k, part size)) is at
//    most the part's kk-th largest logit, hence at most the row's k-th
//    largest.  A 4,096-bin histogram of the maxima' keys, bins of width
//    (range of the maxima) / 4,096 counted from the largest, gives the bin of
//    that maximum; thr = the smallest key of the bin, a bound as good as the
//    maximum itself to within one bin.
//  - Every token with key >= thr is listed as (key, token) -- in thread order,
//    not token order -- through one block scan of per-thread hit counts.  A
//    list longer than kFCap sets the part's flag and the row takes the slices.
template <typename T>
__global__ void __launch_bounds__(kFThreads, 2) filter_kernel(
    const T* __restrict__ logits, int64_t ld, int vocab, int k, int nparts,
    uint2* __restrict__ cand, int* __restrict__ count, float2* __restrict__ stats,
    int* __restrict__ ovf) {
  __shared__ int hist[kWin];
  __shared__ int warp_sums[32];
  __shared__ int s_total;
  __shared__ uint32_t s_kmax[kFThreads / 32], s_kmin[kFThreads / 32];
  __shared__ float2 red2[kFThreads / 32];
  __shared__ uint32_t s_thr;
  const int r = blockIdx.x, part = blockIdx.y;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int base = part * kPart;
  const int n = min(kPart, vocab - base);
  const int kk = min(k, n);
  const T* row = logits + int64_t(r) * ld + base;
  constexpr int W = 16 / sizeof(T);
  constexpr int J = kFPer / W;
  constexpr float kL2e = 1.4426950408889634f;
  const bool full = n == kPart;
  float v[kFPer];
  if (full) {
#pragma unroll
    for (int j = 0; j < J; ++j)
      unpack16<T>(__ldg(reinterpret_cast<const uint4*>(row + (j * kFThreads + t) * W)), v + j * W);
  } else {
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int i0 = (j * kFThreads + t) * W;
      if (i0 + W <= n) {
        unpack16<T>(__ldg(reinterpret_cast<const uint4*>(row + i0)), v + j * W);
      } else {
#pragma unroll
        for (int e = 0; e < W; ++e) v[j * W + e] = i0 + e < n ? Elem<T>::to_f(row[i0 + e]) : -INFINITY;
      }
    }
  }
  for (int i = t; i < kWin; i += kFThreads) hist[i] = 0;
  // ---- the thread's (max, sum of exp(x - max)) and its max's key
  float m = max3(v[0], v[1], v[2]);
#pragma unroll
  for (int i = 3; i + 1 < kFPer; i += 2) m = max3(m, v[i], v[i + 1]);
  m = fmaxf(m, v[kFPer - 1]);
  const bool tvalid = t * W < n;  // the thread holds at least one token
  const uint32_t tk = tvalid ? key_of(m) : 0u;
  float sum = 0.f;
  if (m != -INFINITY) {
    const float mb = m * kL2e;
#pragma unroll
    for (int i = 0; i < kFPer; ++i) sum += ex2(fmaf(v[i], kL2e, -mb));
  }
  uint32_t kmax = tk, kmin = tvalid ? tk : 0xFFFFFFFFu;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, off);
    const float so = __shfl_xor_sync(0xffffffffu, sum, off);
    const float mm = fmaxf(m, mo);
    sum = (m == -INFINITY ? 0.f : sum * ex2((m - mm) * kL2e)) +
          (mo == -INFINITY ? 0.f : so * ex2((mo - mm) * kL2e));
    m = mm;
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, off));
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, off));
  }
  if (lane == 0) {
    red2[warp] = make_float2(m, sum);
    s_kmax[warp] = kmax;
    s_kmin[warp] = kmin;
  }
  __syncthreads();
  // ---- thr: the smallest key of the histogram bin that holds the kk-th
  // largest thread maximum (0, every token, when fewer threads hold tokens)
  uint32_t KM = 0u, Km = 0xFFFFFFFFu;
#pragma unroll
  for (int w = 0; w < kFThreads / 32; ++w) {
    KM = max(KM, s_kmax[w]);
    Km = min(Km, s_kmin[w]);
  }
  const int holders = min(kFThreads, (n + W - 1) / W);
  uint32_t thr = 0u;
  if (holders >= kk) {  // uniform over the block
    const uint32_t span = KM - Km;
    const int sh = span < uint32_t(kWin) ? 0 : 20 - __clz(span);  // span >> sh < 4,096
    if (tvalid) atomicAdd(&hist[(KM - tk) >> sh], 1);
    __syncthreads();
    constexpr int per = kWin / kFThreads;
    int c = 0;
#pragma unroll
    for (int q = 0; q < per; ++q) c += hist[t * per + q];
    const int excl = block_scan<kFThreads>(c, warp_sums, &s_total);
    if (excl < kk && kk <= excl + c) {
      int acc = excl, b = t * per;
      for (int q = 0; q < per; ++q) {
        acc += hist[t * per + q];
        if (acc >= kk) {
          b = t * per + q;
          break;
        }
      }
      const int64_t lo = int64_t(KM) - ((int64_t(b) + 1) << sh) + 1;
      s_thr = lo < 0 ? 0u : uint32_t(lo);
    }
    __syncthreads();
    thr = s_thr;
  }
  // ---- the tokens at or above thr (compared as floats: thr_f is the value
  // of key thr, -inf when thr admits every token), counted, placed by a block
  // scan, then written; padding (tail part) never counts
  const float thr_f = thr <= key_of(-INFINITY) ? -INFINITY : value_of(thr);
  int mine = 0;
  if (tvalid && tk >= thr) {
    if (full) {
#pragma unroll
      for (int i = 0; i < kFPer; ++i) mine += v[i] >= thr_f;
    } else {
#pragma unroll
      for (int j = 0; j < J; ++j)
#pragma unroll
        for (int e = 0; e < W; ++e) mine += (j * kFThreads + t) * W + e < n && v[j * W + e] >= thr_f;
    }
  }
  int pos = block_scan<kFThreads>(mine, warp_sums, &s_total);
  const int total = s_total;
  const int64_t slot = int64_t(r) * nparts + part;
  if (total > kFCap || total < kk) {  // uniform: the row takes the slices
    if (t == 0) ovf[slot] = 1;
    return;
  }
  if (mine) {
    uint2* out = cand + slot * kFCap;
#pragma unroll
    for (int j = 0; j < J; ++j)
#pragma unroll
      for (int e = 0; e < W; ++e) {
        const int i = (j * kFThreads + t) * W + e;
        if (v[j * W + e] >= thr_f && (full || i < n))
          out[pos++] = make_uint2(key_of(v[j * W + e]), uint32_t(base + i));
      }
  }
  if (t == 0) {
    float M = -INFINITY, S = 0.f;
    for (int w = 0; w < kFThreads / 32; ++w) M = fmaxf(M, red2[w].x);
    for (int w = 0; w < kFThreads / 32; ++w)
      if (red2[w].x != -INFINITY) S += red2[w].y * ex2((red2[w].x - M) * kL2e);
    stats[slot] = make_float2(M, S);
    count[slot] = total;
    ovf[slot] = 0;
  }
}

// Merge, one CTA per row, over the row's candidates: the parts' lists, or
// (a flagged row) the slices' k each, E per thread (key 0: an empty place).
//  - Window pass: a 4,096-bin histogram of the candidates' keys, bins of
//    width (key range) / 4,096 counted from the largest, and a block scan of
//    it give each bin's first place in the order and the bin b of the k-th
//    largest.  Every candidate of a bin up to b takes its bin's next place in
//    shared memory; its final place is its bin's first place plus the number
//    of words of its bin above its own (64-bit (key, ~token) words: ties go
//    to the smaller token).  Places below k are the row's k, in order.
//  - When bin b and the bins above it hold more than kMergeList candidates
//    (many copies of one logit): an exact radix select of the k-th largest
//    key (12-, 10- and 10-bit passes) and, when that key has more copies than
//    places, of the smallest tokens among them (two 10-bit passes); the k
//    winners are placed by a block scan and sorted bitonically (warp shuffles
//    for strides below 32).
// Then lse from the (max, sum) pairs, p = exp(x - lse) and Z.
constexpr int kMergeList = 2048;

__global__ void __launch_bounds__(kMergeThreads, 1) merge_kernel(
    const uint2* __restrict__ cand8, const float2* __restrict__ stats8, int nslices,
    const uint2* __restrict__ candf, const int* __restrict__ countf,
    const float2* __restrict__ statsf, int nparts, const int* __restrict__ ovf, int vocab, int k,
    int32_t* __restrict__ ids, float* __restrict__ probs, float* __restrict__ z,
    float* __restrict__ lse_out) {
  constexpr int E = kMaxSlices * kMaxK / kMergeThreads;  // candidates per thread
  constexpr int NW = kMergeThreads / 32;
  __shared__ SelectSmem sel;  // its histogram is the window histogram too
  __shared__ unsigned long long wl[kMergeList];
  __shared__ uint32_t s_kmax[NW], s_kmin[NW];
  __shared__ float red[NW];
  __shared__ float s_lse;
  __shared__ int s_b, s_above, s_m;
  const int r = blockIdx.x, t = threadIdx.x, warp = t >> 5, lane = t & 31;
  bool slices = false;
  for (int p = 0; p < nparts; ++p) slices = slices || ovf[int64_t(r) * nparts + p] != 0;
  // ---- the row's normaliser from the (max, sum) pairs
  if (warp == 0) {
    const int nst = slices ? nslices : nparts;
    const float2* st_row = slices ? stats8 + int64_t(r) * nslices : statsf + int64_t(r) * nparts;
    const float2 st = lane < nst ? st_row[lane] : make_float2(-INFINITY, 0.f);
    float M = st.x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float S = st.x == -INFINITY ? 0.f : st.y * expf(st.x - M);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) S += __shfl_xor_sync(0xffffffffu, S, off);
    if (lane == 0) s_lse = M + logf(S);
  }
  // ---- the candidates
  uint32_t key[E], tok[E];
  if (slices) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = t * E + e, sl = i / k, c = i % k;
      key[e] = 0u;
      tok[e] = 0u;
      if (sl < nslices && c < min(k, vocab - sl * kSlice)) {
        const uint2 w = cand8[(int64_t(r) * nslices + sl) * k + c];
        key[e] = w.x;
        tok[e] = w.y;
      }
    }
  } else {
    const int p = (t * E) / kFCap;  // E divides kFCap: one part per thread
    const int n_p = p < nparts ? countf[int64_t(r) * nparts + p] : 0;
    const uint2* src = candf + (int64_t(r) * nparts + p) * kFCap;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int c = (t * E + e) % kFCap;
      key[e] = 0u;
      tok[e] = 0u;
      if (c < n_p) {
        const uint2 w = src[c];
        key[e] = w.x;
        tok[e] = w.y;
      }
    }
  }
  // ---- window histogram over [min, max] of the keys
  for (int i = t; i < 4096; i += kMergeThreads) sel.hist[i] = 0;
  uint32_t kx = 0u, kn = 0xFFFFFFFFu;
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (key[e] != 0u) {
      kx = max(kx, key[e]);
      kn = min(kn, key[e]);
    }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    kx = max(kx, __shfl_xor_sync(0xffffffffu, kx, off));
    kn = min(kn, __shfl_xor_sync(0xffffffffu, kn, off));
  }
  if (lane == 0) {
    s_kmax[warp] = kx;
    s_kmin[warp] = kn;
  }
  __syncthreads();
  uint32_t KM = 0u, Km = 0xFFFFFFFFu;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    KM = max(KM, s_kmax[w]);
    Km = min(Km, s_kmin[w]);
  }
  const uint32_t span = KM - Km;
  const int sh = span < 4096u ? 0 : 20 - __clz(span);  // span >> sh < 4,096
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (key[e] != 0u) atomicAdd(&sel.hist[(KM - key[e]) >> sh], 1);
  __syncthreads();
  constexpr int per = 4096 / kMergeThreads;
  int c[per], cnt = 0;
#pragma unroll
  for (int q = 0; q < per; ++q) {
    c[q] = sel.hist[t * per + q];
    cnt += c[q];
  }
  int acc = block_scan<kMergeThreads>(cnt, sel.warp_sums, &sel.total);
#pragma unroll
  for (int q = 0; q < per; ++q) {  // first places in the order, in place
    if (acc < k && k <= acc + c[q]) {
      s_b = t * per + q;
      s_above = acc;
      s_m = c[q];
    }
    sel.hist[t * per + q] = acc;
    acc += c[q];
  }
  __syncthreads();
  const int b = s_b, placed = s_above + s_m;
  const float L = s_lse;
  float psum = 0.f;
  if (placed <= kMergeList) {  // uniform
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if (key[e] == 0u) continue;
      const int bin = int((KM - key[e]) >> sh);
      if (bin <= b) wl[atomicAdd(&sel.hist[bin], 1)] = sort_word(key[e], tok[e]);
    }
    __syncthreads();
    // a bin's places are now [end of the bin before, its own end)
    for (int q = t; q < placed; q += kMergeThreads) {
      const unsigned long long w = wl[q];
      const uint32_t kq = static_cast<uint32_t>(w >> 32);
      const int bin = int((KM - kq) >> sh);
      const int first = bin ? sel.hist[bin - 1] : 0, last = sel.hist[bin];
      int place = first;
      for (int x = first; x < last; ++x) place += wl[x] > w;
      if (place < k) {
        const float pr = expf(value_of(kq) - L);
        ids[int64_t(r) * k + place] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(w & 0xFFFFFFFFull));
        probs[int64_t(r) * k + place] = pr;
        psum += pr;
      }
    }
  } else {
    // the k winners: keys above thr, and need_eq of the keys equal to it
    // (the smallest tokens), placed by a block scan, then sorted
    int need_eq = 0;
    const uint32_t thr = select_kth<kMergeThreads, E>(key, k, sel, need_eq);
    const int eq_total = sel.bin_cnt;
    uint32_t rank_cut = 0u;  // every copy of thr wins
    if (need_eq < eq_total) rank_cut = select_tok<kMergeThreads, E>(key, tok, thr, need_eq, sel);
    int mine = 0;
#pragma unroll
    for (int e = 0; e < E; ++e)
      mine += key[e] != 0u && (key[e] > thr || (key[e] == thr && kTokRank - tok[e] >= rank_cut));
    int pos = block_scan<kMergeThreads>(mine, sel.warp_sums, &sel.total);
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (key[e] != 0u && (key[e] > thr || (key[e] == thr && kTokRank - tok[e] >= rank_cut)))
        wl[pos++] = sort_word(key[e], tok[e]);
    __syncthreads();
    unsigned long long w = t < k ? wl[t] : 0ull;
    __syncthreads();
    for (int size = 2; size <= kMaxK; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        unsigned long long o;
        if (stride >= 32) {
          if (t < kMaxK) wl[t] = w;
          __syncthreads();
          o = t < kMaxK ? wl[t ^ stride] : 0ull;
          __syncthreads();
        } else {
          o = __shfl_xor_sync(0xffffffffu, w, stride);
        }
        const bool desc = (t & size) == 0, lower = (t & stride) == 0;
        const unsigned long long hi = w > o ? w : o, lo = w > o ? o : w;
        w = (lower == desc) ? hi : lo;
      }
    }
    if (t < k) {
      const float pr = expf(value_of(static_cast<uint32_t>(w >> 32)) - L);
      ids[int64_t(r) * k + t] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(w & 0xFFFFFFFFull));
      probs[int64_t(r) * k + t] = pr;
      psum = pr;
    }
  }
  // ---- Z, the mass of the k
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
  if (lane == 0) red[warp] = psum;
  __syncthreads();
  if (t == 0) {
    float Z = 0.f;
    for (int w2 = 0; w2 < NW; ++w2) Z += red[w2];
    if (z) z[r] = Z;
    if (lse_out) lse_out[r] = L;
  }
}

static int nslices_of(int vocab) { return (vocab + kSlice - 1) / kSlice; }

static int nparts_of(int vocab) { return (vocab + kPart - 1) / kPart; }

// workspace: slice candidates and (max, sum); part lists, their lengths and
// (max, sum); the parts' overflow flags
struct RoLayout {
  size_t cand8, stats8, candf, countf, statsf, ovf, total;
};
static RoLayout ro_layout(int rows, int vocab, int k) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t R = static_cast<size_t>(rows), ns = nslices_of(vocab), np = nparts_of(vocab);
  RoLayout Y;
  Y.cand8 = 0;
  Y.stats8 = al(Y.cand8 + R * ns * k * sizeof(uint2));
  Y.candf = al(Y.stats8 + R * ns * sizeof(float2));
  Y.countf = al(Y.candf + R * np * kFCap * sizeof(uint2));
  Y.statsf = al(Y.countf + R * np * sizeof(int));
  Y.ovf = al(Y.statsf + R * np * sizeof(float2));
  Y.total = al(Y.ovf + R * np * sizeof(int));
  return Y;
}
static size_t ws_bytes_of(int rows, int vocab, int k) { return ro_layout(rows, vocab, k).total; }

static int check_shape(int dtype, int rows, int vocab, int k) {
  if (dtype != PIE_F32 && dtype != PIE_BF16) return set_last_error(PIE_EINVAL, "readout: unknown dtype");
  if (rows < 0 || vocab < 1) return set_last_error(PIE_EINVAL, "readout: need rows >= 0 and vocab >= 1");
  if (k < 1 || k > vocab) return set_last_error(PIE_EINVAL, "readout: need 1 <= k <= vocab");
  if (k > kMaxK) return set_last_error(PIE_EUNSUPPORTED, "readout: k above 256 is not built");
  if (nslices_of(vocab) > kMaxSlices)
    return set_last_error(PIE_EUNSUPPORTED, "readout: vocab above 262,144 is not built");
  return PIE_OK;
}

}  // namespace ro

}  // namespace pie

using namespace pie;

extern "C" int pie_fwd_readout_topk_workspace_bytes(int32_t dtype, int32_t rows, int32_t vocab,
                                                    int32_t k, size_t* bytes) {
  if (!bytes) return set_last_error(PIE_EINVAL, "bytes is NULL");
  const int rc = ro::check_shape(dtype, rows, vocab, k);
  if (rc != PIE_OK) return rc;
  *bytes = ro::ws_bytes_of(rows, vocab, k);
  return PIE_OK;
}

extern "C" int pie_fwd_readout_topk(const void* logits, int32_t dtype, int32_t rows,
                                    int32_t vocab, int64_t ld, int32_t k, int32_t* ids,
                                    float* probs, float* z, float* lse, void* workspace,
                                    size_t ws_bytes, void* stream) {
  const int rc = ro::check_shape(dtype, rows, vocab, k);
  if (rc != PIE_OK) return rc;
  if (rows == 0) return PIE_OK;
  if (!logits || !ids || !probs) return set_last_error(PIE_EINVAL, "readout: logits, ids and probs are required");
  const size_t esize = dtype == PIE_BF16 ? 2 : 4;
  if (ld < vocab) return set_last_error(PIE_EINVAL, "readout: ld below vocab");
  if (reinterpret_cast<uintptr_t>(logits) % 16 != 0 || (static_cast<size_t>(ld) * esize) % 16 != 0)
    return set_last_error(PIE_EINVAL, "readout: logits rows must start on 16-byte boundaries");
  const size_t need = ro::ws_bytes_of(rows, vocab, k);
  if (!workspace || ws_bytes < need)
    return set_last_error(PIE_ENOSPACE, "readout: workspace smaller than pie_fwd_readout_topk_workspace_bytes()");
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return set_last_error(PIE_EINVAL, "readout: workspace must be 256-byte aligned");
  const int ns = ro::nslices_of(vocab), np = ro::nparts_of(vocab);
  char* w = static_cast<char*>(workspace);
  const ro::RoLayout Y = ro::ro_layout(rows, vocab, k);
  uint2* cand8 = reinterpret_cast<uint2*>(w + Y.cand8);
  float2* stats8 = reinterpret_cast<float2*>(w + Y.stats8);
  uint2* candf = reinterpret_cast<uint2*>(w + Y.candf);
  int* countf = reinterpret_cast<int*>(w + Y.countf);
  float2* statsf = reinterpret_cast<float2*>(w + Y.statsf);
  int* ovf = reinterpret_cast<int*>(w + Y.ovf);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t smem1 = sizeof(uint32_t) * (ro::kSlice + ro::kSlice / 32);
  static bool configured = false;
  if (!configured) {
    cudaFuncSetAttribute(ro::slice_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem1));
    cudaFuncSetAttribute(ro::slice_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         int(smem1));
    configured = true;
  }
  // parts filter; rows whose parts overflowed go through the slices; merge
  const dim3 g0(rows, np), g1(rows, ns);
  cudaEvent_t ev0, ev1;
  timing_events(&ev0, &ev1);
  if (ev0) cudaEventRecord(ev0, s);
  if (dtype == PIE_BF16) {
    ro::filter_kernel<__nv_bfloat16><<<g0, ro::kFThreads, 0, s>>>(
        static_cast<const __nv_bfloat16*>(logits), ld, vocab, k, np, candf, countf, statsf, ovf);
    if (ev1) cudaEventRecord(ev1, s);
    ro::slice_kernel<__nv_bfloat16><<<g1, ro::kThreads, smem1, s>>>(
        static_cast<const __nv_bfloat16*>(logits), ld, vocab, k, ns, cand8, stats8, ovf, np);
  } else {
    ro::filter_kernel<float><<<g0, ro::kFThreads, 0, s>>>(
        static_cast<const float*>(logits), ld, vocab, k, np, candf, countf, statsf, ovf);
    if (ev1) cudaEventRecord(ev1, s);
    ro::slice_kernel<float><<<g1, ro::kThreads, smem1, s>>>(
        static_cast<const float*>(logits), ld, vocab, k, ns, cand8, stats8, ovf, np);
  }
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) {
    ro::merge_kernel<<<rows, ro::kMergeThreads, 0, s>>>(cand8, stats8, ns, candf, countf, statsf, np,
                                                        ovf, vocab, k, ids, probs, z, lse);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return set_last_error(PIE_ECUDA, std::string("readout launch: ") + cudaGetErrorString(e));
  return PIE_OK;
}
