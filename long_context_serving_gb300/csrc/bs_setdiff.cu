// a5: set-difference of the selection against the previous step, stand-alone kernel
// ("Technisches Resümee: NOSA", Methodik / 2. System: NOSI: set-difference kernels
// for block swapping). One CTA per unit; both ascending lists are staged in shared
// memory; each element of one list is looked up in the other by binary search and the
// misses are compacted in order, so both outputs come out ascending.
#include "bs_select_impl.cuh"

namespace bsi {
namespace {

constexpr int kDiffThreads = 256;

__global__ void __launch_bounds__(kDiffThreads) setdiff_kernel(bs_dims dims, const int32_t *__restrict__ prev,
                                                               const int32_t *__restrict__ prev_cnt,
                                                               const int32_t *__restrict__ cur,
                                                               const int32_t *__restrict__ cur_cnt,
                                                               int32_t *__restrict__ added,
                                                               int32_t *__restrict__ added_cnt,
                                                               int32_t *__restrict__ removed,
                                                               int32_t *__restrict__ removed_cnt, int32_t *st) {
  extern __shared__ __align__(16) int32_t lists[];
  __shared__ SelShared<kDiffThreads> sh;
  const int cap = dims.max_sel_per_unit;
  const int u = blockIdx.x, tid = threadIdx.x;
  int32_t *sp = lists, *sc = lists + cap;
  const size_t row = static_cast<size_t>(u) * cap;
  const int np = prev_cnt[u], nc = cur_cnt[u];
  if (np < 0 || np > cap || nc < 0 || nc > cap) {
    if (tid == 0) {
      report(st, BS_ERR_CAPACITY);
      added_cnt[u] = 0;
      removed_cnt[u] = 0;
    }
    for (int i = tid; i < cap; i += kDiffThreads) added[row + i] = removed[row + i] = -1;
    return;
  }
  for (int i = tid; i < np; i += kDiffThreads) sp[i] = prev[row + i];
  for (int i = tid; i < nc; i += kDiffThreads) sc[i] = cur[row + i];
  __syncthreads();
  const int na = sorted_diff_into<kDiffThreads>(sc, nc, sp, np, added + row, cap, sh);
  const int nr = sorted_diff_into<kDiffThreads>(sp, np, sc, nc, removed + row, cap, sh);
  if (tid == 0) {
    added_cnt[u] = na;
    removed_cnt[u] = nr;
  }
}

}  // namespace
}  // namespace bsi

extern "C" bs_status bs_block_setdiff(const bs_dims *dims, const int32_t *prev_idx, const int32_t *prev_cnt,
                                      const int32_t *cur_idx, const int32_t *cur_cnt, int32_t *added,
                                      int32_t *added_cnt, int32_t *removed, int32_t *removed_cnt,
                                      int32_t *dev_status, bs_stream_t stream) {
  using namespace bsi;
  bs_status s = check_dims(dims);
  if (s != BS_OK) return s;
  if (!prev_idx || !prev_cnt || !cur_idx || !cur_cnt || !added || !added_cnt || !removed || !removed_cnt ||
      !dev_status)
    return BS_ERR_INVALID_ARG;
  if (dims->max_sel_per_unit > 24576) return BS_ERR_CAPACITY;  // two lists in shared memory
  const int units = dims->batch * dims->n_kv_heads;
  const size_t smem = static_cast<size_t>(dims->max_sel_per_unit) * 2 * sizeof(int32_t);
  static const cudaError_t attr = cudaFuncSetAttribute(
      setdiff_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(24576 * 2 * sizeof(int32_t)));
  if (attr != cudaSuccess) return BS_ERR_CUDA;
  setdiff_kernel<<<units, kDiffThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(
      *dims, prev_idx, prev_cnt, cur_idx, cur_cnt, added, added_cnt, removed, removed_cnt, dev_status);
  return launch_status();
}
