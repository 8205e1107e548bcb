// Attention kernels for bf16 caches (tiled TMA + warp-level tensor-core MMA, device
// code attn_split_mma in bs_attn_impl.cuh) and their launcher.
#include "bs_attn_impl.cuh"
#include "bs_attn_launch.cuh"

namespace bsi {
namespace {

template <int D, int G>
__global__ void __launch_bounds__(kMmaThreads) attn_mma_kernel(AttnArgs a, const __grid_constant__ CUtensorMap tmk,
                                                               const __grid_constant__ CUtensorMap tmv, bool step,
                                                               bool cluster) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  if (step) pdl_launch_dependents();
  const bool took_part = attn_split_mma<D, G>(a, &tmk, &tmv, align_smem_1024(smem_raw), step, cluster);
  // In the fused step, finish only after the selection kernel has (a split that took no
  // part leaves at once: split 0 of every unit takes part, so the grid still does).
  if (step && took_part) pdl_wait();
}

template <int D, int G>
bs_status launch_modes(const AttnArgs &a, bool step, const CUtensorMap &tk, const CUtensorMap &tv, cudaStream_t cs) {
  const int units = a.dims.batch * a.dims.n_kv_heads;
  constexpr int kSmemMax = MmaLayout<D>::bytes(MmaLayout<D>::kRingMax) + kSmemAlignSlack;
  auto kernel = attn_mma_kernel<D, G>;
  static const bool attrs_ok =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax) == cudaSuccess &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
  if (!attrs_ok) return BS_ERR_CUDA;
  const bool cluster = attn_mode(units, a.dims.max_gather_pages_per_unit) == kModeCluster;
  const int smem = MmaLayout<D>::bytes(attn_mma_ring(cluster)) + kSmemAlignSlack;
  const int splits = attn_grid_splits(units, a.dims.max_gather_pages_per_unit, attn_target_ctas());
  const dim3 grid = cluster ? dim3(splits, units) : dim3(units, splits);   // (workspace mode: unit-major)
  const cudaError_t e =
      launch_ex(kernel, grid, kMmaThreads, smem, cs, cluster && splits > 1 ? splits : 0, step, a, tk, tv, step, cluster);
  return e == cudaSuccess ? BS_OK : BS_ERR_CUDA;
}

template <int D>
bs_status dispatch_g(const AttnArgs &a, bool step, const CUtensorMap &tk, const CUtensorMap &tv, cudaStream_t cs) {
  switch (a.dims.n_q_heads / a.dims.n_kv_heads) {
    case 1: return launch_modes<D, 1>(a, step, tk, tv, cs);
    case 2: return launch_modes<D, 2>(a, step, tk, tv, cs);
    case 3: return launch_modes<D, 3>(a, step, tk, tv, cs);
    case 4: return launch_modes<D, 4>(a, step, tk, tv, cs);
    case 5: return launch_modes<D, 5>(a, step, tk, tv, cs);
    case 6: return launch_modes<D, 6>(a, step, tk, tv, cs);
    case 7: return launch_modes<D, 7>(a, step, tk, tv, cs);
    default: return launch_modes<D, 8>(a, step, tk, tv, cs);
  }
}

}  // namespace

bs_status launch_attn_bf16(const AttnArgs &a, bool step, cudaStream_t cs) {
  CUtensorMap tk, tv;
  const bs_status s = make_kv_tensor_maps(a.dims, a.kv, &tk, &tv);
  if (s != BS_OK) return s;
  return a.dims.head_dim == 128 ? dispatch_g<128>(a, step, tk, tv, cs) : dispatch_g<64>(a, step, tk, tv, cs);
}

}  // namespace bsi
