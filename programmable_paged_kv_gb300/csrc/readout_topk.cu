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
// per row at 128K fp32 tokens), so the work is spread over slices:
//   1. slice kernel, grid (rows, slices), 512 threads: a 8,192-token slice of
//      a row into shared memory as order-preserving 32-bit keys (coalesced
//      16-byte loads), the slice's max and sum of exp(x - max), then its k
//      largest keys: a 4,096-bin histogram of the top 12 key bits finds the
//      bucket of the k-th key, the keys in it or above (a few hundred) are
//      copied in token order to a short list, and an exact radix select
//      (12-, 10- and 10-bit passes) over the list yields the k (key, token)
//      candidates -- keys equal to the k-th largest taken smallest token
//      first by a block-wide scan (the select runs over all the slice's keys
//      when ties crowd the bucket past 1,024);
//   2. merge kernel, one CTA per row: the same radix select over the slices'
//      candidates keeps the row's k, a bitonic sort of 64-bit (key, ~token)
//      words orders them (warp shuffles for strides below 32), the slices'
//      (max, sum) merge into lse, and p = exp(x - lse) for the kept tokens
//      and their sum Z follow.
// The top k of a row lie in the union of its slices' top k, so the merge
// sees every token it can return.

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
constexpr int kPart = 65536;             // tokens per part of the streaming kernel
constexpr int kStreamThreads = 1024;
constexpr int kStreamList = 2048;        // list capacity of a part (more: the row takes the slices)
constexpr int kMaxParts = 4;             // vocab <= 262,144
constexpr int kSample = 16;              // one token in kSample feeds the streaming histogram

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
  int total, bin, above;
};

// The kk-th largest of the block's keys (E per thread, held in registers;
// key 0 is padding, below every token): a radix select on bits 31..20 (4,096
// bins: the sign, the exponent and three mantissa bits, so a block's keys
// spread over many bins and the shared-memory adds rarely collide), then
// 19..10 and 9..0 among the keys sharing the prefix chosen so far.  Returns
// the key; need_eq = how many keys equal to it belong to the kk (the others
// are the keys above it).
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
    // thread t takes nbins / NT consecutive bins from the top; a block scan
    // of their counts (top first) finds the bin that holds the rem-th key
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
          break;
        }
        acc += c;
      }
    }
    __syncthreads();
    rem -= sm.above;
    prefix |= uint32_t(sm.bin) << shift;
    pmask |= bmask << shift;
    __syncthreads();  // hist, bin and above are rewritten by the next pass
  }
  need_eq = rem;
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
  // only rows whose streaming parts overflowed their lists come here
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
__device__ __forceinline__ unsigned long long sort_word(uint2 c) {
  return (static_cast<unsigned long long>(c.x) << 32) | (0xFFFFFFFFu - c.y);
}

// Streaming kernel, grid (rows, parts), 1,024 threads: a 65,536-token part of
// a row read twice -- first from HBM for its (max, sum) and a 4,096-bin
// histogram of the top 12 key bits of one token in 16, which gives a bucket
// with about 2k sampled-and-scaled keys at or above it; then again (from L2)
// to list the keys at or above that bucket as 64-bit (key, ~token) words,
// unique per token, so their order does not matter.  A bitonic sort of the
// list (at most 2,048) gives the part's k, largest first.  A part whose list
// holds fewer than its k or overflows (ties, a flat distribution, an unlucky
// sample) sets its flag, and its row goes through the slice kernel instead.
template <typename T>
__global__ void __launch_bounds__(kStreamThreads, 1) stream_kernel(
    const T* __restrict__ logits, int64_t ld, int vocab, int k, int nparts,
    uint2* __restrict__ cand, float2* __restrict__ stats, int* __restrict__ ovf) {
  __shared__ SelectSmem sel;
  __shared__ unsigned long long lst[kStreamList];
  __shared__ float2 red2[kStreamThreads / 32];
  __shared__ int s_count;
  const int r = blockIdx.x, part = blockIdx.y;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int base = part * kPart;
  const int n = min(kPart, vocab - base);
  const int kk = min(k, n);
  const T* row = logits + int64_t(r) * ld + base;
  constexpr int W = 16 / sizeof(T);
  constexpr int kStep = kStreamThreads * W;
  constexpr float kL2e = 1.4426950408889634f;
  const int nchunks = (n + kStep - 1) / kStep;
  for (int i = t; i < 4096; i += kStreamThreads) sel.hist[i] = 0;
  if (t == 0) s_count = 0;
  __syncthreads();
  auto load = [&](int i0, float* f) {
    if (i0 + W <= n) {
      unpack16<T>(*reinterpret_cast<const uint4*>(row + i0), f);
    } else {
#pragma unroll
      for (int e = 0; e < W; ++e) f[e] = i0 + e < n ? Elem<T>::to_f(row[i0 + e]) : -INFINITY;
    }
  };
  // ---- pass 1: online (max, sum of exp(x - max)) and the histogram
  float m = -INFINITY, sum = 0.f;
#pragma unroll 2
  for (int c = 0; c < nchunks; ++c) {
    const int i0 = c * kStep + t * W;
    float f[W];
    load(i0, f);
    float cm = f[0];
#pragma unroll
    for (int e = 1; e < W; ++e) cm = fmaxf(cm, f[e]);
    if (cm > m) {
      sum = m == -INFINITY ? 0.f : sum * ex2((m - cm) * kL2e);
      m = cm;
    }
#pragma unroll
    for (int e = 0; e < W; ++e) {
      if (i0 + e < n) {
        if (m != -INFINITY) sum += ex2((f[e] - m) * kL2e);
        // one token in kSample goes into the histogram: a per-token add
        // into a few crowded bins would cost more than the whole stream
        if (((i0 + e) & (kSample - 1)) == 0) atomicAdd(&sel.hist[key_of(f[e]) >> 20], 1);
      }
    }
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
    for (int w = 0; w < kStreamThreads / 32; ++w) M = fmaxf(M, red2[w].x);
    for (int w = 0; w < kStreamThreads / 32; ++w)
      if (red2[w].x != -INFINITY) S += red2[w].y * ex2((red2[w].x - M) * kL2e);
    stats[int64_t(r) * nparts + part] = make_float2(M, S);
  }
  // ---- a bucket the sample puts about 2 kk keys at or above (at least 4
  // sampled keys); pass 2 counts them exactly
  const int need_s = max(4, (2 * kk + kSample - 1) / kSample);
  int sampled_ge = 0;
  const uint32_t cb = find_bucket<kStreamThreads>(need_s, sel, sampled_ge);
  // ---- pass 2: the keys at or above the bucket, one warp-wide add per hit
  const uint32_t below = (1u << lane) - 1u;
#pragma unroll 2
  for (int c = 0; c < nchunks; ++c) {
    const int i0 = c * kStep + t * W;
    float f[W];
    load(i0, f);
#pragma unroll
    for (int e = 0; e < W; ++e) {
      const uint32_t key = key_of(f[e]);
      const bool hit = i0 + e < n && (key >> 20) >= cb;
      const uint32_t mask = __ballot_sync(0xffffffffu, hit);
      if (mask) {
        const int leader = __ffs(mask) - 1;
        int at = 0;
        if (lane == leader) at = atomicAdd(&s_count, __popc(mask));
        at = __shfl_sync(0xffffffffu, at, leader);
        const int slot = at + __popc(mask & below);
        if (hit && slot < kStreamList)
          lst[slot] = (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - uint32_t(base + i0 + e));
      }
    }
  }
  __syncthreads();
  // the list must hold the part's kk and fit: otherwise the row takes the
  // slices (exact for any distribution)
  const int count_ge = s_count;
  if (count_ge < kk || count_ge > kStreamList) {
    if (t == 0) ovf[int64_t(r) * nparts + part] = 1;
    return;
  }
  if (t == 0) ovf[int64_t(r) * nparts + part] = 0;
  // ---- bitonic sort of the list, largest first.  Up to 1,024 entries: one
  // per thread, strides below 32 by warp shuffles (no barrier), larger ones
  // through shared memory; beyond that, pairs in shared memory throughout.
  int p2 = 2;
  while (p2 < count_ge) p2 <<= 1;
  for (int i = count_ge + t; i < p2; i += kStreamThreads) lst[i] = 0ull;
  __syncthreads();
  if (p2 <= kStreamThreads) {
    unsigned long long v = t < p2 ? lst[t] : 0ull;
    for (int size = 2; size <= p2; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        unsigned long long o;
        if (stride >= 32) {
          __syncthreads();
          if (t < p2) lst[t] = v;
          __syncthreads();
          o = t < p2 ? lst[t ^ stride] : 0ull;
        } else {
          o = __shfl_xor_sync(0xffffffffu, v, stride);
        }
        const bool desc = (t & size) == 0, lower = (t & stride) == 0;
        const unsigned long long hi = v > o ? v : o, lo = v > o ? o : v;
        v = (lower == desc) ? hi : lo;
      }
    }
    __syncthreads();
    if (t < p2) lst[t] = v;
    __syncthreads();
  } else {
  for (int size = 2; size <= p2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = t; i < p2 / 2; i += kStreamThreads) {
        const int lo = 2 * i - (i & (stride - 1)), hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long x = lst[lo], y = lst[hi];
        if ((x < y) == desc) {
          lst[lo] = y;
          lst[hi] = x;
        }
      }
      __syncthreads();
    }
  }
  }
  uint2* out = cand + (int64_t(r) * nparts + part) * k;
  for (int j = t; j < kk; j += kStreamThreads) {
    const unsigned long long w = lst[j];
    out[j] = make_uint2(static_cast<uint32_t>(w >> 32), 0xFFFFFFFFu - static_cast<uint32_t>(w & 0xFFFFFFFFull));
  }
}

// Merge, one CTA per row.  Rows whose parts streamed: each part's k are
// sorted, so a candidate's place in the row is its index in its part plus,
// for every other part, the number of that part's candidates above it (a
// binary search); places below k are the row's k, already in order.  Rows
// that went through the slices: the radix select over the slices'
// candidates, then a bitonic sort of the k (warp shuffles for strides below
// 32).  Then lse from the (max, sum) pairs, p = exp(x - lse) and Z.
__global__ void __launch_bounds__(kMergeThreads, 1) merge_kernel(
    const uint2* __restrict__ cand8, const float2* __restrict__ stats8, int nslices,
    const uint2* __restrict__ cand64, const float2* __restrict__ stats64, int nparts,
    const int* __restrict__ ovf, int vocab, int k, int32_t* __restrict__ ids,
    float* __restrict__ probs, float* __restrict__ z, float* __restrict__ lse_out) {
  constexpr int E = kMaxSlices * kMaxK / kMergeThreads;  // candidates per thread
  __shared__ SelectSmem sel;
  __shared__ uint2 win[kMaxK];
  __shared__ unsigned long long xs[kMaxK];
  __shared__ unsigned long long pw[kMaxParts][kMaxK];
  __shared__ float red[kMergeThreads / 32];
  __shared__ float s_lse;
  const int r = blockIdx.x, t = threadIdx.x, warp = t >> 5, lane = t & 31;
  bool slices = false;
  for (int p = 0; p < nparts; ++p) slices = slices || ovf[int64_t(r) * nparts + p] != 0;
  // ---- the row's normaliser from the (max, sum) pairs
  if (warp == 0) {
    const int nst = slices ? nslices : nparts;
    const float2* st_row = slices ? stats8 + int64_t(r) * nslices : stats64 + int64_t(r) * nparts;
    const float2 st = lane < nst ? st_row[lane] : make_float2(-INFINITY, 0.f);
    float M = st.x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float S = st.x == -INFINITY ? 0.f : st.y * expf(st.x - M);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) S += __shfl_xor_sync(0xffffffffu, S, off);
    if (lane == 0) s_lse = M + logf(S);
  }
  unsigned long long w = 0ull;
  if (!slices) {
    for (int i = t; i < nparts * kMaxK; i += kMergeThreads) {
      const int p = i / kMaxK, j = i % kMaxK;
      pw[p][j] = j < min(k, vocab - p * kPart) ? sort_word(cand64[(int64_t(r) * nparts + p) * k + j]) : 0ull;
    }
    __syncthreads();
    for (int i = t; i < nparts * kMaxK; i += kMergeThreads) {
      const int p = i / kMaxK, j = i % kMaxK;
      if (j >= min(k, vocab - p * kPart)) continue;
      const unsigned long long x = pw[p][j];
      int place = j;
      for (int q = 0; q < nparts; ++q) {
        if (q == p) continue;
        int lo = 0, hi = min(k, vocab - q * kPart);
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (pw[q][mid] > x) lo = mid + 1;
          else hi = mid;
        }
        place += lo;
      }
      if (place < k) xs[place] = x;
    }
    __syncthreads();
    w = t < k ? xs[t] : 0ull;
  } else {
  uint32_t key[E], tok[E];
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
  // ---- the k winners (unordered), then a bitonic sort of them, largest
  // first, one per thread of the first eight warps: strides below 32 by warp
  // shuffles, larger strides through shared memory
  int need_eq = 0;
  const uint32_t thr = select_kth<kMergeThreads, E>(key, k, sel, need_eq);
  emit_selected<kMergeThreads, E>(key, TokList<E>{tok}, thr, need_eq, sel, win);
  __syncthreads();
  w = (t < k) ? sort_word(win[t]) : 0ull;
  for (int size = 2; size <= kMaxK; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      unsigned long long o;
      if (stride >= 32) {
        if (t < kMaxK) xs[t] = w;
        __syncthreads();
        o = t < kMaxK ? xs[t ^ stride] : 0ull;
        __syncthreads();
      } else {
        o = __shfl_xor_sync(0xffffffffu, w, stride);
      }
      const bool desc = (t & size) == 0, lower = (t & stride) == 0;
      const unsigned long long hi = w > o ? w : o, lo = w > o ? o : w;
      w = (lower == desc) ? hi : lo;
    }
  }
  }
  // ---- tokens, p, and their mass
  const float L = s_lse;
  float p = 0.f;
  if (t < k) {
    const float x = value_of(static_cast<uint32_t>(w >> 32));
    p = expf(x - L);
    ids[int64_t(r) * k + t] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(w & 0xFFFFFFFFull));
    probs[int64_t(r) * k + t] = p;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
  if (lane == 0) red[warp] = p;
  __syncthreads();
  if (t == 0) {
    float Z = 0.f;
    for (int w2 = 0; w2 < kMergeThreads / 32; ++w2) Z += red[w2];
    if (z) z[r] = Z;
    if (lse_out) lse_out[r] = L;
  }
}

static int nslices_of(int vocab) { return (vocab + kSlice - 1) / kSlice; }

static int nparts_of(int vocab) { return (vocab + kPart - 1) / kPart; }

// workspace: slice candidates and (max, sum), part candidates and (max, sum),
// the parts' overflow flags
struct RoLayout {
  size_t cand8, stats8, cand64, stats64, ovf, total;
};
static RoLayout ro_layout(int rows, int vocab, int k) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t R = static_cast<size_t>(rows), ns = nslices_of(vocab), np = nparts_of(vocab);
  RoLayout Y;
  Y.cand8 = 0;
  Y.stats8 = al(Y.cand8 + R * ns * k * sizeof(uint2));
  Y.cand64 = al(Y.stats8 + R * ns * sizeof(float2));
  Y.stats64 = al(Y.cand64 + R * np * k * sizeof(uint2));
  Y.ovf = al(Y.stats64 + R * np * sizeof(float2));
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
  uint2* cand64 = reinterpret_cast<uint2*>(w + Y.cand64);
  float2* stats64 = reinterpret_cast<float2*>(w + Y.stats64);
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
  // parts stream; rows whose parts overflowed go through the slices; merge
  const dim3 g0(rows, np), g1(rows, ns);
  if (dtype == PIE_BF16) {
    ro::stream_kernel<__nv_bfloat16><<<g0, ro::kStreamThreads, 0, s>>>(
        static_cast<const __nv_bfloat16*>(logits), ld, vocab, k, np, cand64, stats64, ovf);
    ro::slice_kernel<__nv_bfloat16><<<g1, ro::kThreads, smem1, s>>>(
        static_cast<const __nv_bfloat16*>(logits), ld, vocab, k, ns, cand8, stats8, ovf, np);
  } else {
    ro::stream_kernel<float><<<g0, ro::kStreamThreads, 0, s>>>(
        static_cast<const float*>(logits), ld, vocab, k, np, cand64, stats64, ovf);
    ro::slice_kernel<float><<<g1, ro::kThreads, smem1, s>>>(
        static_cast<const float*>(logits), ld, vocab, k, ns, cand8, stats8, ovf, np);
  }
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) {
    ro::merge_kernel<<<rows, ro::kMergeThreads, 0, s>>>(cand8, stats8, ns, cand64, stats64, np, ovf,
                                                        vocab, k, ids, probs, z, lse);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return set_last_error(PIE_ECUDA, std::string("readout launch: ") + cudaGetErrorString(e));
  return PIE_OK;
}
