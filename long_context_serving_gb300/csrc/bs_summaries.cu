// a1: sub-block mean keys (first stage of NOSA's two-stage pooling, "Technisches
// Resümee: NOSA", Methodik / 1. Algorithmus: NOSA, "Blockweise Implementierung";
// NOSI fuses this pooling with the KV write, "2. System: NOSI").
//
// One warp per sub-block; lane l owns head_dim/32 consecutive dimensions. Tokens are
// summed in token order in fp32 and divided by the number present, so an update of
// one sub-block gives the same bits as a full rebuild.
#include "bs_internal.cuh"

namespace bsi {
namespace {

constexpr int kSumThreads = 128;

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

template <int D, typename KT>
__global__ void __launch_bounds__(kSumThreads) summaries_kernel(bs_dims dims, bs_kv kv, bs_head_cfg cfg,
                                                                const int32_t *__restrict__ tok_begin,
                                                                float *__restrict__ summ, int32_t *st) {
  constexpr int DPL = D / 32;
  const int u = blockIdx.y;
  const int b = u / dims.n_kv_heads;
  const int T = kv.seq_lens[b];
  const int g = cfg.block_tokens[u], s = cfg.sub_tokens[u];
  if (!unit_cfg_ok(cfg.cls[u], g, s, cfg.k_total[u], cfg.k_evict[u], cfg.sink_tokens[u],
                   cfg.local_tokens[u])) {
    if (threadIdx.x == 0) report(st, BS_ERR_INVALID_ARG);
    return;
  }
  int begin = tok_begin[b];
  if (T < 1 || begin < 0 || begin > T) {
    if (threadIdx.x == 0) report(st, BS_ERR_INVALID_ARG);
    return;
  }
  if (begin == T) return;  // nothing appended
  if ((T + kPage - 1) / kPage > dims.max_pages_per_unit) {
    if (threadIdx.x == 0) report(st, BS_ERR_CAPACITY);
    return;
  }
  const int j0 = begin / s, j1 = (T - 1) / s;
  const int64_t off = cfg.sum_off[u];
  if (j1 >= cfg.sum_rows[u] || off < 0) {
    if (threadIdx.x == 0) report(st, BS_ERR_CAPACITY);
    return;
  }
  const int32_t *pt = kv.page_table + static_cast<size_t>(u) * dims.max_pages_per_unit;
  const KT *pool = static_cast<const KT *>(kv.k_pool);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = kSumThreads / 32;
  for (int j = j0 + blockIdx.x * kWarps + warp; j <= j1; j += gridDim.x * kWarps) {
    const int lo = j * s, hi = min((j + 1) * s, T);
    float acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.0f;
    bool bad = false;
    // One page at a time: one page-table load, then every row of the page in flight
    // together; the adds stay in token order.
    for (int t0 = lo; t0 < hi;) {
      const int page_end = min(hi, (t0 / kPage + 1) * kPage);
      const int phys = __ldg(pt + t0 / kPage);
      if (phys < 0 || phys >= dims.n_pages) {
        bad = true;
        break;
      }
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
    if (bad) {
      if (lane == 0) report(st, BS_ERR_DEVICE_BOUNDS);
      continue;
    }
    const float n = static_cast<float>(hi - lo);
    float *dst = summ + off + static_cast<int64_t>(j) * D + lane * DPL;
#pragma unroll
    for (int i = 0; i < DPL; ++i) dst[i] = acc[i] / n;
  }
}

}  // namespace
}  // namespace bsi

extern "C" bs_status bs_build_block_summaries(const bs_dims *dims, const bs_kv *kv, const bs_head_cfg *cfg,
                                              const int32_t *tok_begin, int32_t max_new_tokens,
                                              float *summaries, int32_t *dev_status, bs_stream_t stream) {
  using namespace bsi;
  bs_status s = check_dims(dims);
  if (s != BS_OK) return s;
  if (!kv || !cfg || !kv->k_pool || !kv->page_table || !kv->seq_lens || !cfg->cls || !cfg->block_tokens ||
      !cfg->sub_tokens || !cfg->k_total || !cfg->k_evict || !cfg->sink_tokens || !cfg->local_tokens ||
      !cfg->sum_off || !cfg->sum_rows || !tok_begin || !summaries || !dev_status)
    return BS_ERR_INVALID_ARG;
  if (max_new_tokens < 1) return BS_ERR_INVALID_ARG;
  if (!aligned16(kv->k_pool) || !aligned16(summaries)) return BS_ERR_ALIGN;
  const int units = dims->batch * dims->n_kv_heads;
  const int warps = kSumThreads / 32;
  int gx = (max_new_tokens + 1 + warps - 1) / warps;
  if (gx > 4096) gx = 4096;
  const dim3 grid(gx, units);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (dims->head_dim == 128 && dims->kv_dtype == BS_BF16)
    summaries_kernel<128, uint16_t><<<grid, kSumThreads, 0, cs>>>(*dims, *kv, *cfg, tok_begin, summaries, dev_status);
  else if (dims->head_dim == 128)
    summaries_kernel<128, float><<<grid, kSumThreads, 0, cs>>>(*dims, *kv, *cfg, tok_begin, summaries, dev_status);
  else if (dims->kv_dtype == BS_BF16)
    summaries_kernel<64, uint16_t><<<grid, kSumThreads, 0, cs>>>(*dims, *kv, *cfg, tok_begin, summaries, dev_status);
  else
    summaries_kernel<64, float><<<grid, kSumThreads, 0, cs>>>(*dims, *kv, *cfg, tok_begin, summaries, dev_status);
  return launch_status();
}
