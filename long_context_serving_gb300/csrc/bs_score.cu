// a2: block scores, the second stage of NOSA's two-stage pooling ("Technisches
// Resümee: NOSA", Methodik / 1. Algorithmus: NOSA, "Blockweise Implementierung":
// max pooling at block level), shared by the query heads of a GQA group
// ("Technische Samenvatting: Fluxion", Systeemcomponenten, "Granularity-Budget
// Selector").
//
// One CTA per tile of 64 consecutive summary rows (64/r whole blocks, r = g/s) of
// one unit. The tile arrives in shared memory with one bulk copy; four threads share
// a row, each taking every fourth 16-byte chunk in a row-rotated order so that the
// 8 lanes of a shared-memory phase hit 8 different bank groups. The G query vectors
// (pre-scaled by 1/sqrt(d)) sit in shared memory and are read as broadcasts.
#include <math.h>

#include "bs_internal.cuh"

namespace bsi {
namespace {

constexpr int kScoreThreads = 256;
constexpr int kTileRows = 64;

template <int D, int G>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(bs_dims dims, const void *__restrict__ q,
                                                              bs_head_cfg cfg, const int32_t *__restrict__ seq_lens,
                                                              const float *__restrict__ summ, int reduce,
                                                              float *__restrict__ scores, int32_t *st) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ uint64_t bar;
  float *tile = reinterpret_cast<float *>(smem_raw);  // [64][D]
  float *qs = tile + kTileRows * D;                      // [G][D]
  float *dots = qs + G * D;                              // [64][G]

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
  const int r = g / s;           // sub-blocks per block (power of two <= 64)
  const int bpt = kTileRows / r; // whole blocks per tile
  const int c_first = ge.c_lo + blockIdx.x * bpt;
  if (c_first >= ge.c_hi) return;
  const int nb = min(bpt, ge.c_hi - c_first);
  const int nrows = nb * r;
  const int64_t row0 = static_cast<int64_t>(c_first) * r;

  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t bytes = static_cast<uint32_t>(nrows) * D * sizeof(float);
    mbar_arrive_expect_tx(&bar, bytes);
    bulk_g2s(tile, summ + off + row0 * D, bytes, &bar);
  }
  const float scale = rsqrtf(static_cast<float>(D));
  const size_t qbase = (static_cast<size_t>(b) * dims.n_q_heads + static_cast<size_t>(hk) * G) * D;
  for (int i = tid; i < G * D; i += kScoreThreads) qs[i] = load_scalar(q, qbase + i, dims.q_dtype) * scale;
  const bool ok = mbar_wait_bounded(&bar, 0, st);
  if (__syncthreads_or(!ok)) return;

  // Dot products: thread (row, quarter).
  constexpr int kChunks = D / 4;           // float4 chunks per row
  constexpr int kPer = kChunks / 4;        // chunks per quarter (power of two)
  const int row = tid >> 2, qq = tid & 3;
  float acc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) acc[h] = 0.0f;
  if (row < nrows) {
    const float4 *rp = reinterpret_cast<const float4 *>(tile + row * D);
#pragma unroll
    for (int c = 0; c < kPer; ++c) {
      const int ch = qq + 4 * ((c + row) & (kPer - 1));
      const float4 k4 = rp[ch];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float4 q4 = reinterpret_cast<const float4 *>(qs + h * D)[ch];
        acc[h] = fmaf(q4.x, k4.x, acc[h]);
        acc[h] = fmaf(q4.y, k4.y, acc[h]);
        acc[h] = fmaf(q4.z, k4.z, acc[h]);
        acc[h] = fmaf(q4.w, k4.w, acc[h]);
      }
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 1);
    acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 2);
  }
  if (row < nrows && qq == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) dots[row * G + h] = acc[h];
  }
  __syncthreads();
  // Max over the r sub-blocks of a block per head, then over (or mean across) heads.
  if (tid < nb) {
    float red = reduce == BS_GROUP_MAX ? -INFINITY : 0.0f;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float m = -INFINITY;
      for (int j = 0; j < r; ++j) m = fmaxf(m, dots[(tid * r + j) * G + h]);
      red = reduce == BS_GROUP_MAX ? fmaxf(red, m) : red + m;
    }
    if (reduce != BS_GROUP_MAX) red = red / static_cast<float>(G);
    row_out[c_first + tid] = red;
  }
}

template <int D, int G>
void launch_score(const bs_dims &dims, const void *q, const bs_head_cfg &cfg, const int32_t *seq_lens,
                  const float *summ, int reduce, float *scores, int32_t *st, cudaStream_t cs) {
  const int units = dims.batch * dims.n_kv_heads;
  const dim3 grid(dims.max_subs_per_unit / kTileRows + 2, units);
  const size_t smem = (kTileRows * D + G * D + kTileRows * G) * sizeof(float);
  score_kernel<D, G><<<grid, kScoreThreads, smem, cs>>>(dims, q, cfg, seq_lens, summ, reduce, scores, st);
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
