// a3: per-unit block selection, stand-alone kernel (one CTA of 512 threads per unit).
// The selection itself is select_unit() in bs_select_impl.cuh.
#include "bs_select_impl.cuh"

namespace bsi {
namespace {

constexpr int kSelThreads = 512;

__global__ void __launch_bounds__(kSelThreads) select_kernel(bs_dims dims, bs_head_cfg cfg,
                                                             const int32_t *__restrict__ seq_lens,
                                                             const float *__restrict__ scores,
                                                             const float *__restrict__ evict, uint8_t *alive,
                                                             int32_t *__restrict__ sel_idx,
                                                             int32_t *__restrict__ sel_cnt, int32_t *st) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ SelShared<kSelThreads> sh;
  const int MB = dims.max_blocks_per_unit;
  uint32_t *keys = reinterpret_cast<uint32_t *>(smem_raw);       // [MB]
  uint8_t *flags = reinterpret_cast<uint8_t *>(keys + MB);       // [MB]
  const int u = blockIdx.x, tid = threadIdx.x;
  const int b = u / dims.n_kv_heads;
  int32_t *out = sel_idx + static_cast<size_t>(u) * dims.max_sel_per_unit;

  const int cls = cfg.cls[u], g = cfg.block_tokens[u], s = cfg.sub_tokens[u];
  const int k = cfg.k_total[u], k_e = cfg.k_evict[u];
  const int T = seq_lens[b];
  int code = BS_OK;
  if (!unit_cfg_ok(cls, g, s, k, k_e, cfg.sink_tokens[u], cfg.local_tokens[u]) || T < 1) code = BS_ERR_INVALID_ARG;
  else if (cls == BS_DUAL && (evict == nullptr || alive == nullptr)) code = BS_ERR_INVALID_ARG;
  else if ((T + g - 1) / g > MB) code = BS_ERR_CAPACITY;
  if (code != BS_OK) {
    if (tid == 0) {
      report(st, code);
      sel_cnt[u] = 0;
    }
    for (int i = tid; i < dims.max_sel_per_unit; i += kSelThreads) out[i] = -1;
    return;
  }
  const size_t row = static_cast<size_t>(u) * MB;
  SelUnit su;
  su.cls = cls;
  su.k = k;
  su.k_e = k_e;
  su.ge = unit_geom(T, g, s, cfg.sink_tokens[u], cfg.local_tokens[u]);
  su.scores = scores + row;
  su.evict = cls == BS_DUAL ? evict + row : nullptr;
  su.alive = cls == BS_DUAL ? alive + row : nullptr;
  const int total = select_unit<kSelThreads>(su, keys, flags, out, dims.max_sel_per_unit, nullptr, sh);
  if (tid == 0) {
    if (total < 0) report(st, BS_ERR_CAPACITY);
    sel_cnt[u] = total < 0 ? 0 : total;
  }
}

}  // namespace
}  // namespace bsi

extern "C" bs_status bs_select_topk(const bs_dims *dims, const bs_head_cfg *cfg, const int32_t *seq_lens,
                                    const float *scores, const float *evict_logits, uint8_t *alive,
                                    int32_t *sel_idx, int32_t *sel_cnt, int32_t *dev_status,
                                    bs_stream_t stream) {
  using namespace bsi;
  bs_status s = check_dims(dims);
  if (s != BS_OK) return s;
  if (!cfg || !seq_lens || !scores || !sel_idx || !sel_cnt || !dev_status || !cfg->cls || !cfg->block_tokens ||
      !cfg->sub_tokens || !cfg->k_total || !cfg->k_evict || !cfg->sink_tokens || !cfg->local_tokens)
    return BS_ERR_INVALID_ARG;
  const int units = dims->batch * dims->n_kv_heads;
  const size_t smem = static_cast<size_t>(dims->max_blocks_per_unit) * 5;
  static const cudaError_t attr = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       static_cast<int>(kMaxBlocks * 5));
  if (attr != cudaSuccess) return BS_ERR_CUDA;
  select_kernel<<<units, kSelThreads, (smem + 15) & ~size_t(15), reinterpret_cast<cudaStream_t>(stream)>>>(
      *dims, *cfg, seq_lens, scores, evict_logits, alive, sel_idx, sel_cnt, dev_status);
  return launch_status();
}
