// Step 1 of a ForwardPass (Pie "The forward pass", State geometry: each row
// carries an explicit position ID for RoPE and a slot of its lane's working
// set where its K/V state is written).
//
// One CTA per row, or gridDim.y CTAs per row for passes of few rows (a decode
// step's 64 rows would otherwise leave most SMs idle and each CTA several
// dependent load rounds).  Each CTA evaluates the row's D/2 rotation angles
// positions[r] * base^(-2i/d) once into shared memory (fp32 angle, CUDA's
// accurate sincosf) and reuses them for its share of the row's q and k heads.
// Work is split into 16-byte units so that every global load and store is one
// coalesced vector access:
//   * a rotation unit covers VEC elements of the low half [i, i+VEC) and the
//     matching VEC elements of the high half [i+d/2, ...) of one head;
//   * a copy unit moves VEC elements of one v head into the pool.
// K/V go to page page_ids[page_indptr[lane] + slot / P] at offset slot % P
// of the [page][kv head][slot][d] pools.

#include "common.cuh"

namespace pie {

template <typename T, int D>
__global__ void __launch_bounds__(128) rope_scatter_kernel(
    DevMeta m, int Hq, int Hkv, int P, const T* q, const T* k, const T* v, T* q_rot,
    T* k_pool, T* v_pool, const int32_t* frozen_len, uint32_t* status) {
  constexpr int VEC = 16 / sizeof(T);
  constexpr int HALF_UNITS = D / 2 / VEC;
  constexpr int FULL_UNITS = D / VEC;
  __shared__ float s_cos[D / 2], s_sin[D / 2];

  // after the kernels before it (in the decode loop, the one that writes this
  // step's geometry); then the attention kernel may start its set-up
  grid_dep_wait();
  grid_dep_launch();
  const int r = blockIdx.x;
  const int pos = m.positions[r];
  const int lane = m.row_lane[r];
  const int slot = m.slots[r];
  for (int i = threadIdx.x; i < D / 2; i += blockDim.x) {
    const float theta = static_cast<float>(pos) * m.rope_freq[i];
    float sn, cs;
    sincosf(theta, &sn, &cs);
    s_cos[i] = cs;
    s_sin[i] = sn;
  }
  const int frozen = frozen_len[lane];
  bool write_kv = slot >= frozen;
  if (threadIdx.x == 0) {
    if (!write_kv && slot >= 0) set_status(status, PIE_STATUS_FROZEN_WRITE);
    if (r == m.row_indptr[lane] && m.fold_mode[lane] != PIE_FOLD_NONE && slot != frozen)
      set_status(status, PIE_STATUS_FOLD_GAP);
  }
  // (a row that writes nothing -- a frozen slot, or none at all -- reads no
  // page; a page id outside the pool, possible where device code supplies the
  // page table, is not written and sets PIE_STATUS_BOUNDS)
  int64_t page = write_kv ? m.page_ids[m.page_indptr[lane] + slot / P] : 0;
  if (write_kv && (page < 0 || page >= m.num_pool_pages)) {
    if (threadIdx.x == 0) set_status(status, PIE_STATUS_BOUNDS);
    write_kv = false;
    page = 0;
  }
  const int64_t slot_off = page * Hkv * P + (slot % P);  // (page, head 0, slot) in rows of D
  __syncthreads();

  const int q_units = Hq * HALF_UNITS;
  const int k_units = write_kv ? Hkv * HALF_UNITS : 0;
  const int v_units = write_kv ? Hkv * FULL_UNITS : 0;
  const int total = q_units + k_units + v_units;
  // this CTA's units: every gridDim.y-th run of blockDim.x units
  const int stride = blockDim.x * gridDim.y;
  for (int u = blockIdx.y * blockDim.x + threadIdx.x; u < total; u += stride) {
    if (u < q_units + k_units) {
      const bool is_q = u < q_units;
      const int uu = is_q ? u : u - q_units;
      const int h = uu / HALF_UNITS, c = uu % HALF_UNITS;
      const T* src = is_q ? q + (static_cast<int64_t>(r) * Hq + h) * D
                          : k + (static_cast<int64_t>(r) * Hkv + h) * D;
      T* dst = is_q ? q_rot + (static_cast<int64_t>(r) * Hq + h) * D
                    : k_pool + (slot_off + static_cast<int64_t>(h) * P) * D;
      const int i0 = c * VEC;
      float lo[VEC], hi[VEC], olo[VEC], ohi[VEC];
      unpack16<T>(*reinterpret_cast<const uint4*>(src + i0), lo);
      unpack16<T>(*reinterpret_cast<const uint4*>(src + D / 2 + i0), hi);
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float cs = s_cos[i0 + e], sn = s_sin[i0 + e];
        olo[e] = lo[e] * cs - hi[e] * sn;
        ohi[e] = hi[e] * cs + lo[e] * sn;
      }
      *reinterpret_cast<uint4*>(dst + i0) = pack16<T>(olo);
      *reinterpret_cast<uint4*>(dst + D / 2 + i0) = pack16<T>(ohi);
    } else {
      const int uu = u - q_units - k_units;
      const int g = uu / FULL_UNITS, c = uu % FULL_UNITS;
      const T* src = v + (static_cast<int64_t>(r) * Hkv + g) * D + c * VEC;
      T* dst = v_pool + (slot_off + static_cast<int64_t>(g) * P) * D + c * VEC;
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
    }
  }
}

template <typename T, int D>
static cudaError_t launch_rs(const pie_fwd_plan_t& p, const void* q, const void* k, const void* v,
                             void* q_rot, void* k_pool, void* v_pool, const int32_t* frozen,
                             uint32_t* status, cudaStream_t s) {
  // few rows (decode): split each row's units over 4 CTAs
  const dim3 grid(p.N, p.N < 256 ? 4 : 1);
  return launch_dependent(rope_scatter_kernel<T, D>, grid, dim3(128), 0, s, true, p.dev,
                          p.desc.num_q_heads, p.desc.num_kv_heads, p.desc.page_size,
                          static_cast<const T*>(q), static_cast<const T*>(k),
                          static_cast<const T*>(v), static_cast<T*>(q_rot), static_cast<T*>(k_pool),
                          static_cast<T*>(v_pool), frozen, status);
}

cudaError_t launch_rope_scatter(const pie_fwd_plan_t& p, const void* q, const void* k,
                                const void* v, void* q_rot, void* k_pool, void* v_pool,
                                const int32_t* frozen_len, uint32_t* status, cudaStream_t s) {
  const bool bf = p.desc.dtype == PIE_BF16;
  if (p.desc.head_dim == 128)
    return bf ? launch_rs<__nv_bfloat16, 128>(p, q, k, v, q_rot, k_pool, v_pool, frozen_len, status, s)
              : launch_rs<float, 128>(p, q, k, v, q_rot, k_pool, v_pool, frozen_len, status, s);
  return bf ? launch_rs<__nv_bfloat16, 64>(p, q, k, v, q_rot, k_pool, v_pool, frozen_len, status, s)
            : launch_rs<float, 64>(p, q, k, v, q_rot, k_pool, v_pool, frozen_len, status, s);
}

// ---------------------------------------------------------------------------
// Step 4 (State geometry: fold).  One thread per lane:
//   k = 0 | n | fold_count | clamp(channel, 0, n);  frozen_len += k.
// ---------------------------------------------------------------------------
__global__ void fold_kernel(DevMeta m, int L, int32_t* frozen_len, const int32_t* channel,
                            uint32_t* status) {
  grid_dep_wait();  // the kernels before it, channel included
  grid_dep_launch();
  const int l = blockIdx.x * blockDim.x + threadIdx.x;
  if (l >= L) return;
  const int n = m.row_indptr[l + 1] - m.row_indptr[l];
  int k = 0;
  switch (m.fold_mode[l]) {
    case PIE_FOLD_ALL: k = n; break;
    case PIE_FOLD_COUNT: k = m.fold_count[l]; break;
    case PIE_FOLD_CHANNEL: {
      const int c = channel[l];
      k = min(max(c, 0), n);
      if (k != c) set_status(status, PIE_STATUS_FOLD_CLAMP);
      break;
    }
    default: k = 0;
  }
  frozen_len[l] += k;
}

cudaError_t launch_fold(const pie_fwd_plan_t& p, int32_t* frozen_len, const int32_t* channel,
                        uint32_t* status, cudaStream_t s) {
  return launch_dependent(fold_kernel, dim3((p.L + 127) / 128), dim3(128), 0, s, true, p.dev, p.L,
                          frozen_len, channel, status);
}

}  // namespace pie
