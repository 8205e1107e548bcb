// a1: sub-block mean keys, stand-alone kernel: every sub-block that holds a token of
// [tok_begin, T) is recomputed, one warp per sub-block (summary_update_warp() in
// bs_summaries_impl.cuh).
#include "bs_summaries_impl.cuh"

namespace bsi {
namespace {

constexpr int kSumThreads = 128;

template <int D, typename KT>
__global__ void __launch_bounds__(kSumThreads) summaries_kernel(bs_dims dims, bs_kv kv, bs_head_cfg cfg,
                                                                const int32_t *__restrict__ tok_begin,
                                                                float *__restrict__ summ, int32_t *st) {
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
    if (!summary_update_warp<D, KT>(pool, pt, dims.n_pages, s, T, j, summ + off + static_cast<int64_t>(j) * D)) {
      if (lane == 0) report(st, BS_ERR_DEVICE_BOUNDS);
    }
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
