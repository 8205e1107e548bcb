// a2: block scores, stand-alone kernel. One CTA per 64-row tile of a unit's candidate
// summaries (score_tile() in bs_score_impl.cuh); tile 0 also writes -inf to every
// entry of the row outside the candidate range.
#include "bs_score_impl.cuh"

namespace bsi {
namespace {

template <int D, int G>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(bs_dims dims, const void *__restrict__ q,
                                                              bs_head_cfg cfg, const int32_t *__restrict__ seq_lens,
                                                              const float *__restrict__ summ, int reduce,
                                                              float *__restrict__ scores, int32_t *st) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ uint64_t bar;
  const int u = blockIdx.y;
  const int b = u / dims.n_kv_heads, hk = u % dims.n_kv_heads;
  const int tid = threadIdx.x;
  const int cls = cfg.cls[u];
  if (cls == BS_STREAMING) return;
  const int g = cfg.block_tokens[u], s = cfg.sub_tokens[u];
  if (!unit_cfg_ok(cls, g, s, cfg.k_total[u], cfg.k_evict[u], cfg.sink_tokens[u], cfg.local_tokens[u])) {
    if (tid == 0 && blockIdx.x == 0) report(st, BS_ERR_INVALID_ARG);
    return;
  }
  const int T = seq_lens[b];
  if (T < 1) {
    if (tid == 0 && blockIdx.x == 0) report(st, BS_ERR_INVALID_ARG);
    return;
  }
  const Geom ge = unit_geom(T, g, s, cfg.sink_tokens[u], cfg.local_tokens[u]);
  const int n_sub = (T + s - 1) / s;
  const int64_t off = cfg.sum_off[u];
  if (ge.n_blk > dims.max_blocks_per_unit || n_sub > cfg.sum_rows[u] || off < 0) {
    if (tid == 0 && blockIdx.x == 0) report(st, BS_ERR_CAPACITY);
    return;
  }
  if (off % 4 != 0) {
    if (tid == 0 && blockIdx.x == 0) report(st, BS_ERR_ALIGN);
    return;
  }
  float *row_out = scores + static_cast<size_t>(u) * dims.max_blocks_per_unit;
  if (blockIdx.x == 0) {
    for (int c = tid; c < dims.max_blocks_per_unit; c += kScoreThreads)
      if (c < ge.c_lo || c >= ge.c_hi) row_out[c] = -INFINITY;
  }
  if (static_cast<int>(blockIdx.x) >= score_tiles(ge)) return;
  const size_t qbase = (static_cast<size_t>(b) * dims.n_q_heads + static_cast<size_t>(hk) * G) * D;
  const void *qrow = dims.q_dtype == BS_BF16 ? static_cast<const void *>(static_cast<const uint16_t *>(q) + qbase)
                                              : static_cast<const void *>(static_cast<const float *>(q) + qbase);
  score_tile<D, G>(summ + off, qrow, dims.q_dtype, ge, blockIdx.x, reduce, row_out, smem_raw, &bar, st);
}

template <int D, int G>
void launch_score(const bs_dims &dims, const void *q, const bs_head_cfg &cfg, const int32_t *seq_lens,
                  const float *summ, int reduce, float *scores, int32_t *st, cudaStream_t cs) {
  const int units = dims.batch * dims.n_kv_heads;
  const dim3 grid(dims.max_subs_per_unit / kTileRows + 2, units);
  score_kernel<D, G><<<grid, kScoreThreads, ScoreLayout<D, G>::kBytes, cs>>>(dims, q, cfg, seq_lens, summ, reduce,
                                                                           scores, st);
}

template <int D>
void dispatch_g(int G, const bs_dims &dims, const void *q, const bs_head_cfg &cfg, const int32_t *seq_lens,
                const float *summ, int reduce, float *scores, int32_t *st, cudaStream_t cs) {
  switch (G) {
    case 1: launch_score<D, 1>(dims, q, cfg, seq_lens, summ, reduce, scores, st, cs); break;
    case 2: launch_score<D, 2>(dims, q, cfg, seq_lens, summ, reduce, scores, st, cs); break;
    case 3: launch_score<D, 3>(dims, q, cfg, seq_lens, summ, reduce, scores, st, cs); break;
    case 4: launch_score<D, 4>(dims, q, cfg, seq_lens, summ, reduce, scores, st, cs); break;
    case 5: launch_score<D, 5>(dims, q, cfg, seq_lens, summ, reduce, scores, st, cs); break;
    case 6: launch_score<D, 6>(dims, q, cfg, seq_lens, summ, reduce, scores, st, cs); break;
    case 7: launch_score<D, 7>(dims, q, cfg, seq_lens, summ, reduce, scores, st, cs); break;
    default: launch_score<D, 8>(dims, q, cfg, seq_lens, summ, reduce, scores, st, cs); break;
  }
}

}  // namespace
}  // namespace bsi

extern "C" bs_status bs_score_blocks(const bs_dims *dims, const void *q, const bs_head_cfg *cfg,
                                     const int32_t *seq_lens, const float *summaries,
                                     bs_group_reduce group_reduce, float *scores, int32_t *dev_status,
                                     bs_stream_t stream) {
  using namespace bsi;
  bs_status s = check_dims(dims);
  if (s != BS_OK) return s;
  if (!q || !cfg || !seq_lens || !summaries || !scores || !dev_status || !cfg->cls || !cfg->block_tokens ||
      !cfg->sub_tokens || !cfg->k_total || !cfg->k_evict || !cfg->sink_tokens || !cfg->local_tokens ||
      !cfg->sum_off || !cfg->sum_rows)
    return BS_ERR_INVALID_ARG;
  if (group_reduce != BS_GROUP_MAX && group_reduce != BS_GROUP_MEAN) return BS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(summaries)) return BS_ERR_ALIGN;
  const int G = dims->n_q_heads / dims->n_kv_heads;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (dims->head_dim == 128)
    dispatch_g<128>(G, *dims, q, *cfg, seq_lens, summaries, group_reduce, scores, dev_status, cs);
  else
    dispatch_g<64>(G, *dims, q, *cfg, seq_lens, summaries, group_reduce, scores, dev_status, cs);
  return launch_status();
}
