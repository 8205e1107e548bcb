// Device code of the sub-block key summaries (a1), shared by the stand-alone kernel and
// the fused decode step: the first stage of NOSA's two-stage pooling ("Technisches
// Resümee: NOSA", Methodik / 1. Algorithmus: NOSA, "Blockweise Implementierung"; NOSI
// fuses this pooling with the KV write, "2. System: NOSI").
//
// One warp per sub-block; lane l owns head_dim/32 consecutive dimensions. Tokens are
// summed in token order in fp32 and divided by the number present, so an update of one
// sub-block gives the same bits as a full rebuild.
#pragma once

#include "bs_internal.cuh"

namespace bsi {

template <int DPL, typename KT>
__device__ __forceinline__ void load_lane(const KT *p, float (&v)[DPL]);

template <>
__device__ __forceinline__ void load_lane<4, uint16_t>(const uint16_t *p, float (&v)[4]) {
  const uint2 w = *reinterpret_cast<const uint2 *>(p);
  v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
}
template <>
__device__ __forceinline__ void load_lane<2, uint16_t>(const uint16_t *p, float (&v)[2]) {
  const uint32_t w = *reinterpret_cast<const uint32_t *>(p);
  v[0] = bf16lo(w); v[1] = bf16hi(w);
}
template <>
__device__ __forceinline__ void load_lane<4, float>(const float *p, float (&v)[4]) {
  const float4 w = *reinterpret_cast<const float4 *>(p);
  v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
}
template <>
__device__ __forceinline__ void load_lane<2, float>(const float *p, float (&v)[2]) {
  const float2 w = *reinterpret_cast<const float2 *>(p);
  v[0] = w.x; v[1] = w.y;
}

// Recomputes sub-block j of a unit (tokens [j*s, min((j+1)*s, T))) into dst_row.
// Called by all 32 lanes of one warp. Returns false (and writes nothing) when a page
// index is outside the pool.
template <int D, typename KT>
__device__ bool summary_update_warp(const KT *pool, const int32_t *pt, int64_t n_pages, int s, int T, int j,
                                    float *dst_row) {
  constexpr int DPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int lo = j * s, hi = min((j + 1) * s, T);
  float acc[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) acc[i] = 0.0f;
  // One page at a time: one page-table load, then every row of the page in flight
  // together; the adds stay in token order.
  for (int t0 = lo; t0 < hi;) {
    const int page_end = min(hi, (t0 / kPage + 1) * kPage);
    const int phys = __ldg(pt + t0 / kPage);
    if (phys < 0 || phys >= n_pages) return false;
    const KT *base = pool + static_cast<size_t>(phys) * kPage * D + lane * DPL;
    float v[kPage][DPL];
#pragma unroll
    for (int r = 0; r < kPage; ++r) {
      const int t = (t0 & ~(kPage - 1)) + r;
      if (t >= t0 && t < page_end) load_lane<DPL, KT>(base + r * D, v[r]);
    }
#pragma unroll
    for (int r = 0; r < kPage; ++r) {
      const int t = (t0 & ~(kPage - 1)) + r;
      if (t >= t0 && t < page_end) {
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] += v[r][i];
      }
    }
    t0 = page_end;
  }
  const float n = static_cast<float>(hi - lo);
  float *dst = dst_row + lane * DPL;
#pragma unroll
  for (int i = 0; i < DPL; ++i) dst[i] = acc[i] / n;
  return true;
}

}  // namespace bsi
