// a4: sparse decode attention over the selected blocks, stand-alone kernels. The
// device code (split-KV flash-decode over TMA-staged pages with an in-kernel LSE
// merge) is in bs_attn_impl.cuh: attn_split_mma for bf16 caches, attn_split_ffma for
// fp32 caches.
#include "bs_attn_impl.cuh"

namespace bsi {
namespace {

template <int D, int G>
__global__ void __launch_bounds__(kMmaThreads) attn_mma_kernel(bs_dims dims, const void *__restrict__ q, bs_kv kv,
                                                               bs_head_cfg cfg, const __grid_constant__ CUtensorMap tmk,
                                                               const __grid_constant__ CUtensorMap tmv,
                                                               const int32_t *__restrict__ sel_idx,
                                                               const int32_t *__restrict__ sel_cnt,
                                                               int32_t *__restrict__ arrivals, float *__restrict__ ws,
                                                               float *__restrict__ out, float *__restrict__ lse,
                                                               int32_t *st) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  attn_split_mma<D, G, false>(dims, q, kv, cfg, &tmk, &tmv, sel_idx, sel_cnt, arrivals, ws, out, lse, st,
                              align_smem_1024(smem_raw));
}

template <int D, int G>
__global__ void __launch_bounds__(kFfmaThreads) attn_ffma_kernel(bs_dims dims, const void *__restrict__ q, bs_kv kv,
                                                                 bs_head_cfg cfg, const int32_t *__restrict__ sel_idx,
                                                                 const int32_t *__restrict__ sel_cnt,
                                                                 int32_t *__restrict__ arrivals,
                                                                 float *__restrict__ ws, float *__restrict__ out,
                                                                 float *__restrict__ lse, int32_t *st) {
  extern __shared__ __align__(128) unsigned char smem[];
  attn_split_ffma<D, G, false>(dims, q, kv, cfg, sel_idx, sel_cnt, arrivals, ws, out, lse, st, smem);
}

template <int D, int G>
bs_status launch_attn(const bs_dims &dims, const void *q, const bs_kv &kv, const bs_head_cfg &cfg,
                      const int32_t *sel_idx, const int32_t *sel_cnt, float *out, float *lse, float *ws,
                      int32_t *st, cudaStream_t cs) {
  const int units = dims.batch * dims.n_kv_heads;
  const dim3 grid(attn_grid_splits(dims.max_gather_pages_per_unit), units);
  int32_t *arrivals = reinterpret_cast<int32_t *>(ws) + units;   // second counter of each unit
  float *records = ws + attn_counter_floats(units);
  if (dims.kv_dtype == BS_BF16) {
    constexpr int kSmem = MmaLayout<D>::kBytes + kSmemAlignSlack;
    static const cudaError_t attr =
        cudaFuncSetAttribute(attn_mma_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (attr != cudaSuccess) return BS_ERR_CUDA;
    CUtensorMap tk, tv;
    const bs_status s = make_kv_tensor_maps(dims, kv, &tk, &tv);
    if (s != BS_OK) return s;
    attn_mma_kernel<D, G><<<grid, kMmaThreads, kSmem, cs>>>(dims, q, kv, cfg, tk, tv, sel_idx, sel_cnt, arrivals,
                                                            records, out, lse, st);
  } else {
    constexpr int kSmem = FfmaLayout<D, G>::kBytes;
    static const cudaError_t attr =
        cudaFuncSetAttribute(attn_ffma_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (attr != cudaSuccess) return BS_ERR_CUDA;
    attn_ffma_kernel<D, G><<<grid, kFfmaThreads, kSmem, cs>>>(dims, q, kv, cfg, sel_idx, sel_cnt, arrivals, records,
                                                              out, lse, st);
  }
  return launch_status();
}

template <int D>
bs_status dispatch_g(int G, const bs_dims &dims, const void *q, const bs_kv &kv, const bs_head_cfg &cfg,
                     const int32_t *sel_idx, const int32_t *sel_cnt, float *out, float *lse, float *ws,
                     int32_t *st, cudaStream_t cs) {
  switch (G) {
    case 1: return launch_attn<D, 1>(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, ws, st, cs);
    case 2: return launch_attn<D, 2>(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, ws, st, cs);
    case 3: return launch_attn<D, 3>(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, ws, st, cs);
    case 4: return launch_attn<D, 4>(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, ws, st, cs);
    case 5: return launch_attn<D, 5>(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, ws, st, cs);
    case 6: return launch_attn<D, 6>(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, ws, st, cs);
    case 7: return launch_attn<D, 7>(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, ws, st, cs);
    default: return launch_attn<D, 8>(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, ws, st, cs);
  }
}

}  // namespace
}  // namespace bsi

extern "C" bs_status bs_sparse_decode_attn(const bs_dims *dims, const void *q, const bs_kv *kv,
                                           const bs_head_cfg *cfg, const int32_t *sel_idx, const int32_t *sel_cnt,
                                           float *out, float *lse, void *workspace, size_t workspace_bytes,
                                           int32_t *dev_status, bs_stream_t stream) {
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
  const int G = dims->n_q_heads / dims->n_kv_heads;
  float *ws = static_cast<float *>(workspace);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (dims->head_dim == 128)
    return dispatch_g<128>(G, *dims, q, *kv, *cfg, sel_idx, sel_cnt, out, lse, ws, dev_status, cs);
  return dispatch_g<64>(G, *dims, q, *kv, *cfg, sel_idx, sel_cnt, out, lse, ws, dev_status, cs);
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
                                                   const int32_t *sel_cnt, float *out, float *lse,
                                                   int32_t *dev_status, bs_stream_t stream) {
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
  const int G = dims->n_q_heads / dims->n_kv_heads;
  float *ws = static_cast<float *>(scratch);
  if (dims->head_dim == 128)
    return dispatch_g<128>(G, *dims, q, *kv, *cfg, sel_idx, sel_cnt, out, lse, ws, dev_status, cs);
  return dispatch_g<64>(G, *dims, q, *kv, *cfg, sel_idx, sel_cnt, out, lse, ws, dev_status, cs);
}
