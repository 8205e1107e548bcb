// Attention kernels for fp32 caches (1-D bulk copies + FFMA, device code
// attn_split_ffma in bs_attn_impl.cuh) and their launcher.
#include "bs_attn_impl.cuh"
#include "bs_attn_launch.cuh"

namespace bsi {
namespace {

template <int D, int G>
__global__ void __launch_bounds__(kFfmaThreads) attn_ffma_kernel(AttnArgs a, bool step, bool cluster) {
  extern __shared__ __align__(128) unsigned char smem[];
  if (step) pdl_launch_dependents();
  const bool took_part = attn_split_ffma<D, G>(a, smem, step, cluster);
  if (step && took_part) pdl_wait();   // (as in the bf16 kernel)
}

template <int D, int G>
bs_status launch_modes(const AttnArgs &a, bool step, cudaStream_t cs) {
  constexpr int kSmem = FfmaLayout<D, G>::kBytes;
  auto kernel = attn_ffma_kernel<D, G>;
  static const bool attrs_ok =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) == cudaSuccess &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
  if (!attrs_ok) return BS_ERR_CUDA;
  const int units = a.dims.batch * a.dims.n_kv_heads;
  const bool cluster = attn_mode(units, a.dims.max_gather_pages_per_unit) == kModeCluster;
  const int splits = attn_grid_splits(units, a.dims.max_gather_pages_per_unit, attn_target_ctas());
  const dim3 grid = cluster ? dim3(splits, units) : dim3(units, splits);   // (workspace mode: unit-major)
  const cudaError_t e =
      launch_ex(kernel, grid, kFfmaThreads, kSmem, cs, cluster && splits > 1 ? splits : 0, step, a, step, cluster);
  return e == cudaSuccess ? BS_OK : BS_ERR_CUDA;
}

template <int D>
bs_status dispatch_g(const AttnArgs &a, bool step, cudaStream_t cs) {
  switch (a.dims.n_q_heads / a.dims.n_kv_heads) {
    case 1: return launch_modes<D, 1>(a, step, cs);
    case 2: return launch_modes<D, 2>(a, step, cs);
    case 3: return launch_modes<D, 3>(a, step, cs);
    case 4: return launch_modes<D, 4>(a, step, cs);
    case 5: return launch_modes<D, 5>(a, step, cs);
    case 6: return launch_modes<D, 6>(a, step, cs);
    case 7: return launch_modes<D, 7>(a, step, cs);
    default: return launch_modes<D, 8>(a, step, cs);
  }
}

}  // namespace

bs_status launch_attn_f32(const AttnArgs &a, bool step, cudaStream_t cs) {
  return a.dims.head_dim == 128 ? dispatch_g<128>(a, step, cs) : dispatch_g<64>(a, step, cs);
}

}  // namespace bsi
