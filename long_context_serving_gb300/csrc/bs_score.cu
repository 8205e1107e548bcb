// a2: block scores, stand-alone kernel. Each CTA scores one or several 64-row tiles of
// a unit's candidate summaries (the tile device code of bs_score_impl.cuh; several tiles
// stream through two buffers); the unit's first CTA also writes -inf to every entry of
// the row outside the candidate range.
#include <algorithm>

#include "bs_score_impl.cuh"

namespace bsi {
namespace {

int score_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 148;
    cached[dev] = sms;
  }
  return cached[dev];
}

template <int D, int G>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(bs_dims dims, const void *__restrict__ q,
                                                              bs_head_cfg cfg, const int32_t *__restrict__ seq_lens,
                                                              const float *__restrict__ summ, int reduce,
                                                              float *__restrict__ scores, int32_t *st, int tpc) {
  using L = ScoreLayout<D, G>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ uint64_t bars[2];
  const int u = blockIdx.y, cj = blockIdx.x;
  const int b = u / dims.n_kv_heads, hk = u % dims.n_kv_heads;
  const int tid = threadIdx.x;
  const int nbuf = tpc > 1 ? 2 : 1;
  const int cls = cfg.cls[u];
  if (cls == BS_STREAMING) return;
  const int g = cfg.block_tokens[u], s = cfg.sub_tokens[u];
  if (!unit_cfg_ok(cls, g, s, cfg.k_total[u], cfg.k_evict[u], cfg.sink_tokens[u], cfg.local_tokens[u])) {
    if (tid == 0 && cj == 0) report(st, BS_ERR_INVALID_ARG);
    return;
  }
  const int T = seq_lens[b];
  if (T < 1) {
    if (tid == 0 && cj == 0) report(st, BS_ERR_INVALID_ARG);
    return;
  }
  const Geom ge = unit_geom(T, g, s, cfg.sink_tokens[u], cfg.local_tokens[u]);
  const int n_sub = (T + s - 1) / s;
  const int64_t off = cfg.sum_off[u];
  if (ge.n_blk > dims.max_blocks_per_unit || n_sub > cfg.sum_rows[u] || off < 0) {
    if (tid == 0 && cj == 0) report(st, BS_ERR_CAPACITY);
    return;
  }
  if (off % 4 != 0) {
    if (tid == 0 && cj == 0) report(st, BS_ERR_ALIGN);
    return;
  }
  float *row_out = scores + static_cast<size_t>(u) * dims.max_blocks_per_unit;
  if (cj == 0) {
    for (int c = tid; c < dims.max_blocks_per_unit; c += kScoreThreads)
      if (c < ge.c_lo || c >= ge.c_hi) row_out[c] = -INFINITY;
  }
  const int t0 = cj * tpc;
  const int my_tiles = max(0, min(tpc, score_tiles(ge) - t0));
  if (my_tiles == 0) return;
  // Tile t covers rows c_lo * r + 64 t onwards; the copies end at the last candidate row.
  const int r = g / s;
  const int64_t row_end = static_cast<int64_t>(ge.c_hi) * r;
  auto tile_row = [&](int t) -> int64_t { return static_cast<int64_t>(ge.c_lo) * r + static_cast<int64_t>(t) * kTileRows; };
  const float *summ_u = summ + off;
  score_bars_init(bars, nbuf);
  __syncthreads();
  int inflight[2] = {0, 0}, uses[2] = {0, 0};
  for (int i = 0; i < nbuf && i < my_tiles; ++i)
    inflight[i] = score_copy<D>(summ_u, tile_row(t0 + i), row_end, smem_raw + i * L::kTileBytes, &bars[i]);
  const size_t qbase = (static_cast<size_t>(b) * dims.n_q_heads + static_cast<size_t>(hk) * G) * D;
  const void *qrow = dims.q_dtype == BS_BF16 ? static_cast<const void *>(static_cast<const uint16_t *>(q) + qbase)
                                              : static_cast<const void *>(static_cast<const float *>(q) + qbase);
  float *qs = reinterpret_cast<float *>(smem_raw + L::off_q(nbuf));
  float *dots = reinterpret_cast<float *>(smem_raw + L::off_dots(nbuf));
  score_load_q<D, G>(qs, qrow, dims.q_dtype);
  ScoreQ<D, G> qf;
  for (int kk = 0; kk < my_tiles; ++kk) {
    const int bi = kk % nbuf;
    const int n_rows = inflight[bi];
    const bool ok = score_wait(&bars[bi], static_cast<uint32_t>(uses[bi] & 1), n_rows, st);
    if (n_rows > 0) ++uses[bi];
    inflight[bi] = 0;
    if (!ok) {
      for (int i = 0; i < nbuf; ++i) score_wait(&bars[i], static_cast<uint32_t>(uses[i] & 1), inflight[i], st);
      return;
    }
    if (kk == 0) qf = score_qfrag<D, G>(qs);   // (the wait above was a CTA barrier)
    score_compute<D, G>(reinterpret_cast<const float *>(smem_raw + bi * L::kTileBytes), qf, dots, ge, t0 + kk,
                        reduce, n_rows, row_out, [&] {
                          if (kk + nbuf < my_tiles)
                            inflight[bi] = score_copy<D>(summ_u, tile_row(t0 + kk + nbuf), row_end,
                                                         smem_raw + bi * L::kTileBytes, &bars[bi]);
                        });
  }
}

template <int D, int G>
void launch_score(const bs_dims &dims, const void *q, const bs_head_cfg &cfg, const int32_t *seq_lens,
                  const float *summ, int reduce, float *scores, int32_t *st, cudaStream_t cs) {
  const int units = dims.batch * dims.n_kv_heads;
  // Tiles per CTA as in the fused step: 1 for small launches, up to 8 for large ones.
  const int max_tiles = dims.max_subs_per_unit / kTileRows + 2;
  const long long work = static_cast<long long>(units) * max_tiles;
  const int slots = 2 * score_sm_count();
  const int tpc = static_cast<int>(std::min<long long>(8, std::max<long long>(1, (work + 2 * slots - 1) / (2 * slots))));
  const int nbuf = tpc > 1 ? 2 : 1;
  const int smem = ScoreLayout<D, G>::bytes(nbuf);
  // (a failed attribute call shows up as a failed launch of the two-buffer size)
  static const cudaError_t attr = cudaFuncSetAttribute(
      score_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, ScoreLayout<D, G>::bytes(2));
  (void)attr;
  const dim3 grid((max_tiles + tpc - 1) / tpc, units);
  score_kernel<D, G><<<grid, kScoreThreads, smem, cs>>>(dims, q, cfg, seq_lens, summ, reduce, scores, st, tpc);
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
