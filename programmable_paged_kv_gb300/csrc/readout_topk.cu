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
// per row at 128K fp32 tokens); four kernels, each after the first launched
// to start while the one before drains:
//   1. sample kernel, one CTA per row: a bound T on the row's candidates, the
//      ceil(k / 4)-th largest (at least the 16th) of the logits of every 16th
//      chunk of 128 tokens, to within 1/4,096 of the sample's range (one
//      shared-memory histogram whose bins span [min, max] of the sample).
//      About 16 s tokens reach T for the s-th sampled one (1,024 at k = 256);
//   2. stream kernel, one CTA of 256 threads per 4,096 tokens of a row, no
//      block barrier but one: every logit read once (16-byte loads, 16 per
//      thread in registers); each warp's max and sum of exp(x - max); the
//      tokens at or above T appended to the row's list at places taken by
//      one atomic add per CTA;
//   3. slice kernel, 512 threads, over the (row, slice) units of the rows
//      whose list missed k tokens or passed its 4,096 places (ties, flat or
//      masked rows, an unlucky sample): a 8,192-token slice into shared
//      memory as order-preserving 32-bit keys, its max and sum, then its
//      exact k largest (a 4,096-bin histogram of the top 12 key bits finds
//      the bucket of the k-th key; the keys in it or above are listed in
//      token order and an exact radix select over the list, or over the whole
//      slice when ties crowd the bucket, yields k (key, token) candidates);
//   4. merge kernel, one CTA per row: over the row's candidates (its list, or
//      the slices' k each), a histogram whose 4,096 bins span the
//      candidates' keys places each candidate of the bins down to the one of
//      the k-th largest at its bin's first place plus its rank inside the bin
//      (64-bit (key, ~token) words, so ties go to the smaller token); when
//      those bins hold too many candidates, an exact radix select and a
//      bitonic sort take over.  The (max, sum) pairs merge into lse, and
//      p = exp(x - lse) and Z follow.
// Every token the row can return is a candidate: a list holds every token at
// or above T, and when at least k tokens reach T the row's top k all do; the
// row's top k lie in the union of its slices' top k.

#include <algorithm>
#include <cmath>
#include <string>
#include <type_traits>

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
constexpr int kChunk = 128;              // tokens per chunk of the sample
constexpr int kSampleEvery = 16;         // one chunk in 16 is sampled
constexpr int kSampleThreads = 1024;
constexpr int kSamplePer = 16;           // sampled tokens per thread: vocab <= 262,144
constexpr int kPart = 4096;              // tokens per CTA of the stream kernel
constexpr int kStreamThreads = 256;
constexpr int kStreamPer = kPart / kStreamThreads;  // tokens per thread, in registers
constexpr int kRowCap = 4096;            // candidates a row may list (more: the row takes the slices)
constexpr int kCntStride = 32;           // a row's count on a 128-byte line of its own
static_assert(kRowCap <= kMaxSlices * kMaxK, "the merge holds either candidate set");
static_assert(kSampleThreads * kSamplePer * kSampleEvery >= kMaxSlices * kSlice, "sample covers vocab");

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

// Sample kernel, one CTA per row, 1,024 threads: the bound T of the row's
// candidates and a zeroed candidate count.  The sample is every 16th chunk of
// 128 tokens (chunks 0, 16, 32, ...); T is the smallest key of the bin that
// holds the s-th largest sampled key, s = max(16, ceil(k / 4)), in a 4,096-bin
// histogram whose bins span [min, max] of the sampled keys (0, every token,
// when fewer than s tokens are sampled).  About 16 s tokens of the row reach
// T (1,024 at k = 256), and at least s do: the sampled ones.  Any T is
// correct once at least k tokens reach it, since the row's top k then all do;
// a row with fewer, or with more than kRowCap, takes the slices.
template <typename T>
__global__ void __launch_bounds__(kSampleThreads, 1) sample_kernel(
    const T* logits, int64_t ld, int vocab, int k, uint32_t* thr, int* cnt) {
  __shared__ int hist[4096];
  __shared__ int warp_sums[32];
  __shared__ int s_total;
  __shared__ uint32_t s_kmax[32], s_kmin[32];
  __shared__ uint32_t s_thr;
  const int r = blockIdx.x, t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const T* row = logits + int64_t(r) * ld;
  // after the kernels before it: then the stream kernel may start loading the
  // logits (they were written before this grid got past its wait)
  grid_dep_wait();
  grid_dep_launch();
  for (int i = t; i < 4096; i += kSampleThreads) hist[i] = 0;
  // sampled token i: chunk (i / 128) * 16, offset i % 128 (key 0: none)
  uint32_t key[kSamplePer];
  int have = 0;
  uint32_t kx = 0u, kn = 0xFFFFFFFFu;
#pragma unroll
  for (int e = 0; e < kSamplePer; ++e) {
    const int i = e * kSampleThreads + t;
    const int tok = (i / kChunk) * (kChunk * kSampleEvery) + i % kChunk;
    key[e] = tok < vocab ? max(key_of(Elem<T>::to_f(row[tok])), 1u) : 0u;
    if (key[e]) {
      ++have;
      kx = max(kx, key[e]);
      kn = min(kn, key[e]);
    }
  }
  kx = __reduce_max_sync(0xffffffffu, kx);
  kn = __reduce_min_sync(0xffffffffu, kn);
  have = __reduce_add_sync(0xffffffffu, have);
  if (lane == 0) {
    s_kmax[warp] = kx;
    s_kmin[warp] = kn;
    warp_sums[warp] = have;
  }
  __syncthreads();
  const uint32_t KM = __reduce_max_sync(0xffffffffu, s_kmax[lane]);
  const uint32_t Km = __reduce_min_sync(0xffffffffu, s_kmin[lane]);
  const int nsamp = __reduce_add_sync(0xffffffffu, warp_sums[lane]);
  const int sk = max(16, (k + 3) / 4);
  uint32_t bound = 0u;
  if (nsamp >= sk) {  // uniform
    const uint32_t span = KM - Km;
    const int sh = span < 4096u ? 0 : 20 - __clz(span);  // span >> sh < 4,096
#pragma unroll
    for (int e = 0; e < kSamplePer; ++e)
      if (key[e]) atomicAdd(&hist[(KM - key[e]) >> sh], 1);
    __syncthreads();
    constexpr int per = 4096 / kSampleThreads;
    int c[per], tot = 0;
#pragma unroll
    for (int q = 0; q < per; ++q) {
      c[q] = hist[t * per + q];
      tot += c[q];
    }
    int acc = block_scan<kSampleThreads>(tot, warp_sums, &s_total);
#pragma unroll
    for (int q = 0; q < per; ++q) {
      if (acc < sk && sk <= acc + c[q]) {
        const int64_t lo = int64_t(KM) - ((int64_t(t * per + q) + 1) << sh) + 1;
        s_thr = lo < 0 ? 0u : uint32_t(lo);
      }
      acc += c[q];
    }
    __syncthreads();
    bound = s_thr;
  }
  if (t == 0) {
    thr[r] = bound;
    cnt[r * kCntStride] = 0;
  }
}

// Stream kernel, one CTA per 4,096-token part of a row, 256 threads: thread
// t holds tokens (j * 256 + t) * W + e (j < 16 / W, e < W; W tokens per
// 16-byte load).  Each warp writes its (max, sum of exp(x - max)) for the
// row's normaliser, and the CTA lists its tokens at or above the row's bound
// (compared as floats: the value of key T, -inf when T admits every token)
// at places taken by one atomic add per CTA on the row's count (the warps'
// shares by a scan of their totals); places past kRowCap are not written (the
// count still grows, and the row takes the slices).
// One part of the stream kernel; kFull: a whole 4,096-token part (no token
// index checks), else the row's ragged last part (padding -inf, never listed).
template <bool kFull, typename T>
__device__ __forceinline__ void stream_part(const T* __restrict__ row, int n, int base, int r,
                                            int slot, const uint32_t* thr, int* cnt,
                                            uint2* cand, float2* wstats, int* s_wt, int* s_base) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  constexpr int W = 16 / sizeof(T);
  constexpr int J = kStreamPer / W;
  constexpr float kL2e = 1.4426950408889634f;
  auto live = [&](int j, int e) { return kFull || (j * kStreamThreads + t) * W + e < n; };
  float v[kStreamPer];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int i0 = (j * kStreamThreads + t) * W;
    if (kFull || i0 + W <= n) {
      unpack16<T>(__ldg(reinterpret_cast<const uint4*>(row + i0)), v + j * W);
    } else {
#pragma unroll
      for (int e = 0; e < W; ++e) v[j * W + e] = i0 + e < n ? Elem<T>::to_f(row[i0 + e]) : -INFINITY;
    }
  }
  // ---- the warp's (max, sum): each thread's sum rescaled once to the warp max
  // (the logits were written before the sample kernel got past its wait)
  static_assert(kStreamPer == 16, "the max tree and the four partial sums take 16 tokens");
  const float m = max3(max3(max3(v[0], v[1], v[2]), max3(v[3], v[4], v[5]), max3(v[6], v[7], v[8])),
                       max3(v[9], v[10], v[11]), max3(max3(v[12], v[13], v[14]), v[15], v[15]));
  float sum = 0.f;
  if (m != -INFINITY) {  // four independent partial sums
    const float mb = m * kL2e;
    float p4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kStreamPer; ++i) p4[i & 3] += ex2(fmaf(v[i], kL2e, -mb));
    sum = (p4[0] + p4[1]) + (p4[2] + p4[3]);
  }
  const uint32_t kw = __reduce_max_sync(0xffffffffu, m == -INFINITY ? 0u : key_of(m));
  const float mw = kw == 0u ? -INFINITY : value_of(kw);
  sum = m == -INFINITY ? 0.f : sum * ex2((m - mw) * kL2e);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane == 0) wstats[int64_t(slot) * (kStreamThreads / 32) + warp] = make_float2(mw, sum);
  // the bound and the zeroed count are the sample kernel's
  grid_dep_wait();
  const uint32_t tk = thr[r];
  const float thr_f = tk <= key_of(-INFINITY) ? -INFINITY : value_of(tk);
  // ---- the tokens at or above the bound
  int mine = 0;
  if (m >= thr_f) {
    int c4[4] = {0, 0, 0, 0};
#pragma unroll
    for (int j = 0; j < J; ++j)
#pragma unroll
      for (int e = 0; e < W; ++e) c4[(j * W + e) & 3] += (v[j * W + e] >= thr_f && live(j, e)) ? 1 : 0;
    mine = (c4[0] + c4[1]) + (c4[2] + c4[3]);
  }
  int incl = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) s_wt[warp] = incl;
  __syncthreads();
  int before = 0, total = 0;  // the earlier warps' hits, the CTA's
#pragma unroll
  for (int w = 0; w < kStreamThreads / 32; ++w) {
    const int c = s_wt[w];
    before += w < warp ? c : 0;
    total += c;
  }
  if (t == 0) *s_base = total ? atomicAdd(&cnt[r * kCntStride], total) : 0;
  __syncthreads();
  int pos = *s_base + before + incl - mine;
  if (mine) {
    uint2* out = cand + int64_t(r) * kRowCap;
#pragma unroll
    for (int j = 0; j < J; ++j)
#pragma unroll
      for (int e = 0; e < W; ++e)
        if (v[j * W + e] >= thr_f && live(j, e)) {
          if (pos < kRowCap)
            out[pos] = make_uint2(key_of(v[j * W + e]), uint32_t(base + (j * kStreamThreads + t) * W + e));
          ++pos;
        }
  }
}

template <typename T>
__global__ void __launch_bounds__(kStreamThreads) stream_kernel(
    const T* __restrict__ logits, int64_t ld, int vocab, int nparts, const uint32_t* thr, int* cnt,
    uint2* cand, float2* wstats) {
  __shared__ int s_wt[kStreamThreads / 32], s_base;
  const int u = blockIdx.x, r = u / nparts, part = u % nparts;
  const int base = part * kPart;
  const int n = min(kPart, vocab - base);
  const T* row = logits + int64_t(r) * ld + base;
  if (n == kPart)
    stream_part<true, T>(row, n, base, r, u, thr, cnt, cand, wstats, s_wt, &s_base);
  else
    stream_part<false, T>(row, n, base, r, u, thr, cnt, cand, wstats, s_wt, &s_base);
  grid_dep_launch();
}

// A row takes the slices when its list missed the k or overflowed.
__device__ __forceinline__ bool row_flagged(const int* cnt, int r, int kk) {
  const int c = cnt[r * kCntStride];
  return c < kk || c > kRowCap;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 2) slice_kernel(const T* __restrict__ logits, int64_t ld,
                                                          int vocab, int k, int nslices,
                                                          uint2* cand, float2* stats,
                                                          const int* cnt, int units) {
  extern __shared__ uint32_t keys[];  // spos(kSlice) words
  __shared__ SelectSmem sel;
  __shared__ float2 red2[kThreads / 32];
  __shared__ __align__(16) uint32_t lkey[kListCap];
  __shared__ uint32_t ltok[kListCap];
  __shared__ int s_list[kThreads];
  __shared__ int s_nlist;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  grid_dep_wait();  // the counts are the stream kernel's
  grid_dep_launch();
  // the CTA's units (row, slice) = blockIdx.x + i * gridDim.x (i < kThreads),
  // kept when a part of their row overflowed its list: one flag read each
  if (t == 0) s_nlist = 0;
  __syncthreads();
  {
    const int u = blockIdx.x + t * gridDim.x;
    if (u < units && row_flagged(cnt, u / nslices, min(k, vocab)))
      s_list[atomicAdd(&s_nlist, 1)] = u;
  }
  __syncthreads();
  const int nlist = s_nlist;
  for (int li = 0; li < nlist; ++li) {
    __syncthreads();  // shared memory of the previous unit
    const int r = s_list[li] / nslices, s = s_list[li] % nslices;
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
}

// 64-bit words compared as the sort order: key, then smaller token first.
__device__ __forceinline__ unsigned long long sort_word(uint32_t key, uint32_t tok) {
  return (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - tok);
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
    const uint2* cand8, const float2* stats8, int nslices, const uint2* candr, const int* cnt,
    const float2* wstats, int nparts, int vocab, int k, int32_t* ids, float* probs, float* z,
    float* lse_out) {
  constexpr int E = kMaxSlices * kMaxK / kMergeThreads;  // candidates per thread
  constexpr int NW = kMergeThreads / 32;
  __shared__ SelectSmem sel;  // its histogram is the window histogram too
  __shared__ unsigned long long wl[kMergeList];
  __shared__ uint32_t s_kmax[NW], s_kmin[NW];
  __shared__ float red[NW];
  static_assert(NW == 32, "one warp entry per lane");
  __shared__ float s_lse;
  __shared__ int s_b, s_above, s_m;
  const int r = blockIdx.x, t = threadIdx.x, warp = t >> 5, lane = t & 31;
  grid_dep_wait();  // the lists, counts and slices of the kernels before
  const bool slices = row_flagged(cnt, r, min(k, vocab));
  // ---- the row's normaliser from its (max, sum) pairs, one per thread
  {
    const int np = slices ? nslices : nparts * (kStreamThreads / 32);
    const float2* st_row =
        slices ? stats8 + int64_t(r) * nslices : wstats + int64_t(r) * nparts * (kStreamThreads / 32);
    float M = -INFINITY, S = 0.f;
    for (int i = t; i < np; i += kMergeThreads) {  // rows of 2,048 pairs and more: fold
      const float2 st = st_row[i];
      const float mm = fmaxf(M, st.x);
      if (mm != -INFINITY) S = S * expf(M - mm) + st.y * expf(st.x - mm);
      M = mm;
    }
    const uint32_t kb = __reduce_max_sync(0xffffffffu, M == -INFINITY ? 0u : key_of(M));
    if (lane == 0) s_kmax[warp] = kb;
    __syncthreads();
    const uint32_t kr = __reduce_max_sync(0xffffffffu, s_kmax[lane]);
    const float MR = kr == 0u ? -INFINITY : value_of(kr);
    S = M == -INFINITY ? 0.f : S * expf(M - MR);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) S += __shfl_xor_sync(0xffffffffu, S, off);
    if (lane == 0) red[warp] = S;
    __syncthreads();
    if (warp == 0) {
      float SR = red[lane];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) SR += __shfl_xor_sync(0xffffffffu, SR, off);
      if (lane == 0) s_lse = MR + logf(SR);
    }
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
    const int n_r = cnt[r * kCntStride];  // at most kRowCap here
    const uint2* src = candr + int64_t(r) * kRowCap;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int c = e * kMergeThreads + t;
      key[e] = 0u;
      tok[e] = 0u;
      if (c < n_r) {
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
  int c[per], mine_bins = 0;
#pragma unroll
  for (int q = 0; q < per; ++q) {
    c[q] = sel.hist[t * per + q];
    mine_bins += c[q];
  }
  int acc = block_scan<kMergeThreads>(mine_bins, sel.warp_sums, &sel.total);
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

static int num_sms() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

static int nslices_of(int vocab) { return (vocab + kSlice - 1) / kSlice; }

static int nparts_of(int vocab) { return (vocab + kPart - 1) / kPart; }

// workspace: slice candidates and (max, sum); the rows' candidate lists,
// counts and bounds; the warps' (max, sum) pairs
struct RoLayout {
  size_t cand8, stats8, candr, cnt, thr, wstats, total;
};
static RoLayout ro_layout(int rows, int vocab, int k) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t R = static_cast<size_t>(rows), ns = nslices_of(vocab), np = nparts_of(vocab);
  RoLayout Y;
  Y.cand8 = 0;
  Y.stats8 = al(Y.cand8 + R * ns * k * sizeof(uint2));
  Y.candr = al(Y.stats8 + R * ns * sizeof(float2));
  Y.cnt = al(Y.candr + R * kRowCap * sizeof(uint2));
  Y.thr = al(Y.cnt + R * kCntStride * sizeof(int));
  Y.wstats = al(Y.thr + R * sizeof(uint32_t));
  Y.total = al(Y.wstats + R * np * (kStreamThreads / 32) * sizeof(float2));
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
  uint2* candr = reinterpret_cast<uint2*>(w + Y.candr);
  int* cnt = reinterpret_cast<int*>(w + Y.cnt);
  uint32_t* thr = reinterpret_cast<uint32_t*>(w + Y.thr);
  float2* wstats = reinterpret_cast<float2*>(w + Y.wstats);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t smem1 = sizeof(uint32_t) * (ro::kSlice + ro::kSlice / 32);
  static std::atomic<uint64_t> configured_f{0}, configured_b{0};
  {
    cudaError_t e = set_smem_limit(ro::slice_kernel<float>, int(smem1), configured_f);
    if (e == cudaSuccess) e = set_smem_limit(ro::slice_kernel<__nv_bfloat16>, int(smem1), configured_b);
    if (e != cudaSuccess)
      return set_last_error(PIE_ECUDA, std::string("readout set-up: ") + cudaGetErrorString(e));
  }
  // the rows' bounds from a sample; one pass over the logits lists the
  // candidates; rows whose lists missed or overflowed go through the slices;
  // the merge
  const int units = rows * np;
  const int units1 = rows * ns;
  const int g1 = std::max(std::min(units1, 2 * ro::num_sms()), (units1 + ro::kThreads - 1) / ro::kThreads);
  cudaEvent_t ev0, ev1;
  timing_events(&ev0, &ev1);
  // each kernel after the first starts while the one before drains (it waits
  // for it before reading its results); with timing events between them, in
  // plain stream order
  const bool pdl = ev0 == nullptr;
  auto run = [&](auto* x) -> cudaError_t {
    using T = std::remove_const_t<std::remove_pointer_t<decltype(x)>>;
    cudaError_t e = launch_dependent(ro::sample_kernel<T>, dim3(rows), dim3(ro::kSampleThreads), 0,
                                     s, pdl, x, ld, vocab, k, thr, cnt);
    if (ev0) cudaEventRecord(ev0, s);
    if (e == cudaSuccess)
      e = launch_dependent(ro::stream_kernel<T>, dim3(units), dim3(ro::kStreamThreads), 0, s, pdl, x,
                           ld, vocab, np, thr, cnt, candr, wstats);
    if (ev1) cudaEventRecord(ev1, s);
    if (e == cudaSuccess)
      e = launch_dependent(ro::slice_kernel<T>, dim3(g1), dim3(ro::kThreads), smem1, s, pdl, x, ld,
                           vocab, k, ns, cand8, stats8, cnt, units1);
    if (e == cudaSuccess)
      e = launch_dependent(ro::merge_kernel, dim3(rows), dim3(ro::kMergeThreads), 0, s, pdl, cand8,
                           stats8, ns, candr, cnt, wstats, np, vocab, k, ids, probs, z, lse);
    return e == cudaSuccess ? cudaGetLastError() : e;
  };
  const cudaError_t e = dtype == PIE_BF16 ? run(static_cast<const __nv_bfloat16*>(logits))
                                          : run(static_cast<const float*>(logits));
  if (e != cudaSuccess) return set_last_error(PIE_ECUDA, std::string("readout launch: ") + cudaGetErrorString(e));
  return PIE_OK;
}
