// Host-side parts of the C ABI that launch nothing: status text, shape checks,
// head-configuration checks and workspace sizing.
#include <atomic>
#include <climits>
#include <cstdint>

#include "bs_attn_plan.cuh"
#include "bs_internal.cuh"

namespace bsi {

namespace {
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitNs};
}  // namespace

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

bs_status check_dims(const bs_dims *d) {
  if (d == nullptr) return BS_ERR_INVALID_ARG;
  if (d->batch < 1 || d->n_kv_heads < 1 || d->n_q_heads < 1) return BS_ERR_INVALID_ARG;
  if (d->n_q_heads % d->n_kv_heads != 0) return BS_ERR_SHAPE;
  const int G = d->n_q_heads / d->n_kv_heads;
  if (G > kMaxG) return BS_ERR_SHAPE;
  if (d->head_dim != 64 && d->head_dim != 128) return BS_ERR_SHAPE;
  if (d->page_size != kPage) return BS_ERR_SHAPE;
  if (d->kv_dtype != BS_BF16 && d->kv_dtype != BS_FP32) return BS_ERR_INVALID_ARG;
  if (d->q_dtype != BS_BF16 && d->q_dtype != BS_FP32) return BS_ERR_INVALID_ARG;
  if (d->max_pages_per_unit < 1 || d->max_blocks_per_unit < 1 || d->max_sel_per_unit < 1 ||
      d->max_subs_per_unit < 1 || d->max_gather_pages_per_unit < 1 || d->n_pages < 1)
    return BS_ERR_INVALID_ARG;
  if (d->max_blocks_per_unit > kMaxBlocks) return BS_ERR_CAPACITY;
  // The attention's tensor maps address pool rows (16 per page) with signed 32-bit
  // coordinates: every row must stay below 2^31.
  if (d->n_pages > static_cast<int64_t>(INT32_MAX) / kPage) return BS_ERR_CAPACITY;
  if (static_cast<int64_t>(d->batch) * d->n_kv_heads > (int64_t(1) << 24)) return BS_ERR_CAPACITY;
  return BS_OK;
}

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}
}  // namespace

bs_status make_kv_tensor_maps(const bs_dims &d, const bs_kv &kv, CUtensorMap *tk, CUtensorMap *tv) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return BS_ERR_CUDA;
  const uint64_t rows = static_cast<uint64_t>(d.n_pages) * kPage;
  if (rows > static_cast<uint64_t>(INT32_MAX)) return BS_ERR_CAPACITY;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d.head_dim), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d.head_dim) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kPage)};
  const cuuint32_t estr[2] = {1, 1};
  for (int i = 0; i < 2; ++i) {
    void *base = const_cast<void *>(i == 0 ? kv.k_pool : kv.v_pool);
    CUresult r = enc(i == 0 ? tk : tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return BS_ERR_CUDA;
  }
  return BS_OK;
}

}  // namespace bsi

extern "C" {

bs_status bs_set_wait_limit_ns(uint64_t limit_ns) {
  if (limit_ns < 1000 || limit_ns > 60000000000ull) return BS_ERR_INVALID_ARG;
  bsi::g_wait_limit_ns.store(limit_ns, std::memory_order_relaxed);
  return BS_OK;
}

uint64_t bs_wait_limit_ns(void) { return bsi::wait_limit_ns(); }

const char *bs_status_string(bs_status s) {
  switch (s) {
    case BS_OK: return "ok";
    case BS_ERR_INVALID_ARG: return "invalid argument";
    case BS_ERR_SHAPE: return "unsupported shape";
    case BS_ERR_ALIGN: return "misaligned pointer or offset";
    case BS_ERR_CAPACITY: return "capacity exceeded";
    case BS_ERR_CUDA: return "CUDA launch failed";
    case BS_ERR_DEVICE_BOUNDS: return "device index out of bounds";
    case BS_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

size_t bs_workspace_size(const bs_dims *dims) {
  if (bsi::check_dims(dims) != BS_OK) return 0;
  const int G = dims->n_q_heads / dims->n_kv_heads;
  const size_t units = static_cast<size_t>(dims->batch) * dims->n_kv_heads;
  const int mg = dims->max_gather_pages_per_unit;
  // Cluster mode keeps the split partials on chip: the counters and the fused step's
  // page lists. Workspace mode: the counters and the split records.
  const int mode = bsi::attn_mode(static_cast<int>(units), mg);
  const size_t tail = mode == bsi::kModeCluster ? bsi::attn_plist_ints(units, mg)
                                                : bsi::attn_record_area_floats(units, G, dims->head_dim, mode);
  return (bsi::attn_counter_floats(units) + tail) * sizeof(float);
}

int bs_decode_step_launches(const bs_dims *dims) {
  if (bsi::check_dims(dims) != BS_OK) return 0;
  const int units = dims->batch * dims->n_kv_heads;
  // Scores, selection, attention; or the front kernel (scores and selection) and the
  // attention.
  return bsi::step_selects_apart(units, dims->max_gather_pages_per_unit, dims->max_blocks_per_unit)
             ? 3
             : 2;
}

bs_status bs_check_head_cfg(const bs_dims *dims, const bs_head_cfg *c, const int32_t *seq_lens_host) {
  bs_status st = bsi::check_dims(dims);
  if (st != BS_OK) return st;
  if (c == nullptr || seq_lens_host == nullptr) return BS_ERR_INVALID_ARG;
  if (!c->cls || !c->block_tokens || !c->sub_tokens || !c->k_total || !c->k_evict || !c->sink_tokens ||
      !c->local_tokens || !c->sum_off || !c->sum_rows)
    return BS_ERR_INVALID_ARG;
  for (int b = 0; b < dims->batch; ++b) {
    const int T = seq_lens_host[b];
    if (T < 1) return BS_ERR_INVALID_ARG;
    if ((T + bsi::kPage - 1) / bsi::kPage > dims->max_pages_per_unit) return BS_ERR_CAPACITY;
    for (int h = 0; h < dims->n_kv_heads; ++h) {
      const int u = b * dims->n_kv_heads + h;
      const int g = c->block_tokens[u], s = c->sub_tokens[u];
      if (!bsi::unit_cfg_ok(c->cls[u], g, s, c->k_total[u], c->k_evict[u], c->sink_tokens[u],
                            c->local_tokens[u]))
        return BS_ERR_INVALID_ARG;
      if (c->sum_off[u] < 0) return BS_ERR_INVALID_ARG;
      if (c->sum_off[u] % 4 != 0) return BS_ERR_ALIGN;
      const int n_sub = (T + s - 1) / s, n_blk = (T + g - 1) / g;
      if (n_sub > c->sum_rows[u] || n_sub > dims->max_subs_per_unit) return BS_ERR_CAPACITY;
      if (n_blk > dims->max_blocks_per_unit) return BS_ERR_CAPACITY;
      const bsi::Geom ge = bsi::unit_geom(T, g, s, c->sink_tokens[u], c->local_tokens[u]);
      const int forced = ge.n_sink + (ge.n_blk - (ge.local_lo > ge.n_sink ? ge.local_lo : ge.n_sink));
      int sel = forced + (c->cls[u] == BS_STREAMING ? 0 : c->k_total[u]);
      if (sel > ge.n_blk) sel = ge.n_blk;
      if (sel > dims->max_sel_per_unit) return BS_ERR_CAPACITY;
      if (static_cast<int64_t>(sel) * (g / bsi::kPage) >
          dims->max_gather_pages_per_unit)
        return BS_ERR_CAPACITY;
    }
  }
  return BS_OK;
}

}  // extern "C"
