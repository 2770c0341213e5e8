// The combine step of a ForwardPass (Pie "The forward pass", Readouts):
// merges the split partial softmax states that the attention kernels leave
// per (row block, kv head, chunk) and gathers the readout rows -- and every
// row's output when it is requested.

#include "common.cuh"

namespace pie {

constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// Combine: one warp per (target row, q head).  Targets [0, R) are the readout
// rows (written to out_readout / lse_readout); targets [R, R + N) are all rows
// (out_all / lse_all) when requested.  Merges the chunks' (max, sum, output)
// in the log2 domain; an empty visible set gives o = 0 and lse = -inf.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(128) combine_kernel(DevMeta m, int Hq, int Hkv, int G, int N,
                                                      int R, int with_all, int tc_bn,
                                                      int tables_early, T* out_readout,
                                                      float* lse_readout, T* out_all,
                                                      float* lse_all) {
  constexpr int DPL = D / 32;
  const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int targets = R + (with_all ? N : 0);
  const bool active = gw < targets * Hq;
  // tables_early: the plan's own tables (uploaded before any kernel of the
  // pass ran) are read while the attention kernels still run; tables that
  // device code wrote, and the partial states, only after the wait
  const int tgt = active ? gw / Hq : 0, h = active ? gw % Hq : 0;
  const bool is_ro = tgt < R;
  CombEntry ce{0, -1, 0, 0, -1, 0, 0, 0};
  int row = 0;
  auto read_tables = [&] {
    if (active) {
      row = is_ro ? m.readout[tgt] : tgt - R;
      ce = m.comb[int64_t(m.row_block[row]) * Hkv + h / G];
    }
  };
  if (tables_early) read_tables();
  grid_dep_wait();  // the attention kernels' partial states
  grid_dep_launch();
  if (!tables_early) read_tables();
  if (!active || ce.nchunks < 0) return;  // < 0: written directly by the tensor-core kernel
  const int qi = (row - ce.row0) * G + h % G;
  // a masked block uses as many chunks as its list length gives, for as many
  // waves of items as its kernel's (one on the tensor-core path, three on the
  // split-KV path)
  const int nch = ce.mblock < 0 ? ce.nchunks
                                : masked_chunks((m.list_len[ce.mblock] + tc_bn - 1) / tc_bn,
                                                ce.nchunks, *m.mask_tiles, Hkv,
                                                m.num_sms * ce.waves);
  float o[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) o[e] = 0.f;
  float M = -INFINITY, Ls = 0.f;
  if (nch <= 32) {
    // lane c holds chunk c's (max, sum): the merged max and sum by warp
    // reductions, then the chunks' outputs four at a time, their loads in flight
    // together, each weighted by its lane's factor
    const float2 ml = lane < nch ? m.part_ml[ce.part_base + lane * ce.stride + qi]
                                 : make_float2(-INFINITY, 0.f);
    M = ml.x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float f = M == -INFINITY || ml.x == -INFINITY ? 0.f : ex2(ml.x - M);
    float lp = f * ml.y;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lp += __shfl_xor_sync(0xffffffffu, lp, off);
    Ls = lp;
    if (M != -INFINITY) {
      for (int c0 = 0; c0 < nch; c0 += 4) {
        float po[4][DPL];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = c0 + u;
          if (c < nch) {
            const float* src = m.part_o + int64_t(ce.part_base + c * ce.stride + qi) * D + lane * DPL;
#pragma unroll
            for (int e = 0; e < DPL; ++e) po[u][e] = src[e];
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = c0 + u;
          const float fc = __shfl_sync(0xffffffffu, f, c & 31);
          if (c < nch) {
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[e] = fmaf(fc, po[u][e], o[e]);
          }
        }
      }
    }
  } else {
    for (int c = 0; c < nch; ++c) M = fmaxf(M, m.part_ml[ce.part_base + c * ce.stride + qi].x);
    if (M != -INFINITY) {
      for (int c = 0; c < nch; ++c) {
        const int idx = ce.part_base + c * ce.stride + qi;
        const float2 ml = m.part_ml[idx];
        const float f = ex2(ml.x - M);
        Ls = fmaf(f, ml.y, Ls);
        const float* po = m.part_o + int64_t(idx) * D + lane * DPL;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[e] = fmaf(f, po[e], o[e]);
      }
    }
  }
  const bool empty = !(Ls > 0.f);
  const float inv = empty ? 0.f : 1.f / Ls;
  const float lse = empty ? -INFINITY : (M + log2f(Ls)) * kLn2;
  T* dst = is_ro ? out_readout : out_all;
  float* ldst = is_ro ? lse_readout : lse_all;
  const int64_t orow = is_ro ? tgt : row;
  if (dst) {
    T* d = dst + (orow * Hq + h) * D + lane * DPL;
#pragma unroll
    for (int e = 0; e < DPL; ++e) d[e] = Elem<T>::from_f(o[e] * inv);
  }
  if (ldst && lane == 0) ldst[orow * Hq + h] = lse;
}

template <typename T, int D>
static cudaError_t launch_comb(const pie_fwd_plan_t& p, void* out_readout, float* lse_readout,
                               void* out_all, float* lse_all, cudaStream_t s) {
  const int with_all = (out_all || lse_all) ? 1 : 0;
  const int64_t warps = int64_t(p.R + (with_all ? p.N : 0)) * p.desc.num_q_heads;
  if (warps == 0) return cudaSuccess;
  return launch_dependent(combine_kernel<T, D>, dim3(int((warps + 3) / 4)), dim3(128), 0, s, true,
                          p.dev, p.desc.num_q_heads, p.desc.num_kv_heads, p.G, p.N, p.R, with_all,
                          tc_kv_tile(p.tc_nt), p.device_tables ? 0 : 1,
                          static_cast<T*>(out_readout), lse_readout,
                          static_cast<T*>(out_all), lse_all);
}

cudaError_t launch_combine(const pie_fwd_plan_t& p, void* out_readout, float* lse_readout,
                           void* out_all, float* lse_all, cudaStream_t s) {
  const bool bf = p.desc.dtype == PIE_BF16;
  if (p.desc.head_dim == 128)
    return bf ? launch_comb<__nv_bfloat16, 128>(p, out_readout, lse_readout, out_all, lse_all, s)
              : launch_comb<float, 128>(p, out_readout, lse_readout, out_all, lse_all, s);
  return bf ? launch_comb<__nv_bfloat16, 64>(p, out_readout, lse_readout, out_all, lse_all, s)
            : launch_comb<float, 64>(p, out_readout, lse_readout, out_all, lse_all, s);
}

}  // namespace pie
