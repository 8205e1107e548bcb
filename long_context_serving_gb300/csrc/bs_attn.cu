// a4: sparse decode attention over the selected blocks: the C-ABI entry points. The
// kernels are in bs_attn_bf16.cu (bf16 caches: tiled TMA and tensor-core MMA) and
// bs_attn_f32.cu (fp32 caches), their device code in bs_attn_impl.cuh.
#include "bs_attn_launch.cuh"

namespace bsi {
namespace {

bs_status launch_standalone(const bs_dims *dims, const void *q, const bs_kv *kv, const bs_head_cfg *cfg,
                            const int32_t *sel_idx, const int32_t *sel_cnt, const float *bias, float *out,
                            float *lse, float *ws, int32_t *st, cudaStream_t cs) {
  const int units = dims->batch * dims->n_kv_heads;
  AttnArgs a;
  a.dims = *dims;
  a.q = q;
  a.kv = *kv;
  a.cfg = *cfg;
  a.sel_idx = sel_idx;
  a.sel_cnt = sel_cnt;
  a.bias = bias;
  a.out = out;
  a.lse = lse;
  const StepWords w = step_words(ws, units);
  a.arrivals = w.arrivals;
  a.records = ws + attn_records_offset(units);
  a.plist = nullptr;
  a.pub = nullptr;
  a.expect = nullptr;
  a.st = st;
  a.wait_ns = wait_limit_ns();
  return dims->kv_dtype == BS_BF16 ? launch_attn_bf16(a, false, cs) : launch_attn_f32(a, false, cs);
}

}  // namespace
}  // namespace bsi

extern "C" bs_status bs_sparse_decode_attn(const bs_dims *dims, const void *q, const bs_kv *kv,
                                           const bs_head_cfg *cfg, const int32_t *sel_idx, const int32_t *sel_cnt,
                                           const float *evict_bias, float *out, float *lse, void *workspace,
                                           size_t workspace_bytes, int32_t *dev_status, bs_stream_t stream) {
  using namespace bsi;
  bs_status s = check_dims(dims);
  if (s != BS_OK) return s;
  if (!q || !kv || !cfg || !kv->k_pool || !kv->v_pool || !kv->page_table || !kv->seq_lens || !cfg->block_tokens ||
      !sel_idx || !sel_cnt || !out || !lse || !workspace || !dev_status)
    return BS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv->k_pool) || !aligned16(kv->v_pool) || !aligned16(out) ||
      !aligned16(workspace))
    return BS_ERR_ALIGN;
  if (workspace_bytes < bs_workspace_size(dims)) return BS_ERR_CAPACITY;
  return launch_standalone(dims, q, kv, cfg, sel_idx, sel_cnt, evict_bias, out, lse,
                           static_cast<float *>(workspace), dev_status, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// Attention without a caller-provided workspace.
//
// Some callers cannot hand this library a workspace: a plugin running inside a host
// engine that owns every device allocation and exposes no allocator, or a serving
// loop that forbids cudaMalloc after start-up because it synchronises the device and
// can fail under memory pressure. For them the split records and arrival counters
// live in a fixed array in this library's own device memory. Each GPU that loads the
// library holds the array until the process exits.
// ---------------------------------------------------------------------------
#include <mutex>

namespace bsi {
namespace {

constexpr size_t kFixedScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_fixed_scratch[kFixedScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_fixed_scratch_mu;
void *g_fixed_scratch_addr[kMaxDevices] = {};

// Device address of g_fixed_scratch on the current device. In host code the array's
// name only stands in for the symbol; the address is looked up once per device (with
// that device current) and cached.
bs_status fixed_scratch_address(void **addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_fixed_scratch_mu);
  if (g_fixed_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fixed_scratch) != cudaSuccess || p == nullptr) return BS_ERR_CUDA;
    g_fixed_scratch_addr[dev] = p;
  }
  *addr = g_fixed_scratch_addr[dev];
  return BS_OK;
}

}  // namespace
}  // namespace bsi

extern "C" bs_status bs_sparse_decode_attn_noalloc(const bs_dims *dims, const void *q, const bs_kv *kv,
                                                   const bs_head_cfg *cfg, const int32_t *sel_idx,
                                                   const int32_t *sel_cnt, const float *evict_bias, float *out,
                                                   float *lse, int32_t *dev_status, bs_stream_t stream) {
  using namespace bsi;
  bs_status s = check_dims(dims);
  if (s != BS_OK) return s;
  if (!q || !kv || !cfg || !kv->k_pool || !kv->v_pool || !kv->page_table || !kv->seq_lens || !cfg->block_tokens ||
      !sel_idx || !sel_cnt || !out || !lse || !dev_status)
    return BS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv->k_pool) || !aligned16(kv->v_pool) || !aligned16(out)) return BS_ERR_ALIGN;
  const size_t need = bs_workspace_size(dims);
  if (need > kFixedScratchBytes) return BS_ERR_CAPACITY;
  void *scratch = nullptr;
  s = fixed_scratch_address(&scratch);
  if (s != BS_OK) return s;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // The arrival counters must start at zero; the array keeps whatever the previous
  // call (possibly one that stopped early) left in it.
  const size_t units = static_cast<size_t>(dims->batch) * dims->n_kv_heads;
  if (cudaMemsetAsync(scratch, 0, attn_counter_floats(units) * sizeof(float), cs) != cudaSuccess) return BS_ERR_CUDA;
  return launch_standalone(dims, q, kv, cfg, sel_idx, sel_cnt, evict_bias, out, lse, static_cast<float *>(scratch),
                           dev_status, cs);
}
