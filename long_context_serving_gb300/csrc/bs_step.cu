// The fused decode step of one layer: all five steps of the path in two launches.
//
// Launch 1, step_front_kernel, one CTA per (score tile, unit):
//   * every tile of a retrieval or dual unit scores its candidate blocks (a2);
//   * the last tile of each unit to finish (an integer arrival ticket, one acquire-
//     release atomic per CTA) selects the unit's blocks (a3), writes the selection and
//     its set-difference against the previous step (a5), and recomputes the sub-block
//     holding the token just appended (a1). That sub-block lies in the always-forced
//     tail block, which no score of this step reads, so a1 can follow a2;
//   * a streaming unit has one tile that does the last three.
// Launch 2, the attention (a4) as a programmatic dependent launch: streaming units'
// splits need no selection and run while launch 1 is still working; the other splits
// wait for launch 1 (griddepcontrol.wait) before reading their selection.
//
// Both kernels are programmatic dependents of the work before them in the stream: they
// read only the per-unit head configuration before waiting for it to finish.
#include "bs_attn_impl.cuh"
#include "bs_score_impl.cuh"
#include "bs_select_impl.cuh"
#include "bs_summaries_impl.cuh"

namespace bsi {
namespace {

constexpr int kFrontThreads = 256;
constexpr int kStepMaxSel = 4096;

__host__ __device__ inline size_t front_select_bytes(int max_blocks, int max_sel) {
  const size_t flags = (static_cast<size_t>(max_blocks) + 15) & ~size_t(15);
  return static_cast<size_t>(max_blocks) * 4 + flags + 2 * static_cast<size_t>(max_sel) * 4;
}

template <int D, typename KT, int G>
__global__ void __launch_bounds__(kFrontThreads) step_front_kernel(bs_dims dims, bs_kv kv, bs_head_cfg cfg,
                                                                   bs_step_io io, int reduce, int32_t *arrivals) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t bar;
  __shared__ SelShared<kFrontThreads> sh;
  __shared__ int is_last;
  const int u = blockIdx.y, tile = blockIdx.x, tid = threadIdx.x;
  const int b = u / dims.n_kv_heads, hk = u % dims.n_kv_heads;
  const int MB = dims.max_blocks_per_unit, MS = dims.max_sel_per_unit;
  int32_t *st = io.dev_status;
  // Per-unit head configuration: read before the preceding work has finished.
  const int cls = cfg.cls[u], g = cfg.block_tokens[u], s = cfg.sub_tokens[u];
  const int k = cfg.k_total[u], k_e = cfg.k_evict[u], sink = cfg.sink_tokens[u], local = cfg.local_tokens[u];
  const int64_t off = cfg.sum_off[u];
  const int rows = cfg.sum_rows[u];
  pdl_wait();                // q, lengths, KV pages, summaries and selection state are now final
  pdl_launch_dependents();   // the attention may start launching

  const int T = kv.seq_lens[b];
  const size_t srow = static_cast<size_t>(u) * MS;
  int code = BS_OK;
  if (!unit_cfg_ok(cls, g, s, k, k_e, sink, local) || T < 1) code = BS_ERR_INVALID_ARG;
  else if (cls == BS_DUAL && (io.evict_logits == nullptr || io.alive == nullptr)) code = BS_ERR_INVALID_ARG;
  else if ((T + g - 1) / g > MB || (T + s - 1) / s > rows || off < 0 ||
           (T + kPage - 1) / kPage > dims.max_pages_per_unit)
    code = BS_ERR_CAPACITY;
  else if (off % 4 != 0) code = BS_ERR_ALIGN;
  if (code != BS_OK) {
    if (tile == 0) {
      if (tid == 0) {
        report(st, code);
        io.cur_cnt[u] = 0;
        io.added_cnt[u] = 0;
        io.removed_cnt[u] = 0;
      }
      for (int i = tid; i < MS; i += kFrontThreads) io.cur_idx[srow + i] = io.added[srow + i] = io.removed[srow + i] = -1;
    }
    return;
  }
  const Geom ge = unit_geom(T, g, s, sink, local);
  int n_tiles = 1;
  if (cls != BS_STREAMING) n_tiles = max(1, score_tiles(ge));
  if (tile >= n_tiles) return;

  float *score_row = io.scores + static_cast<size_t>(u) * MB;
  if (cls != BS_STREAMING && ge.c_hi > ge.c_lo) {
    const size_t qbase = (static_cast<size_t>(b) * dims.n_q_heads + static_cast<size_t>(hk) * G) * D;
    const void *qrow = dims.q_dtype == BS_BF16
                           ? static_cast<const void *>(static_cast<const uint16_t *>(io.q) + qbase)
                           : static_cast<const void *>(static_cast<const float *>(io.q) + qbase);
    if (!score_tile<D, G>(io.summaries + off, qrow, dims.q_dtype, ge, tile, reduce, score_row, smem, &bar, st))
      return;
  }
  if (n_tiles > 1) {
    __syncthreads();
    if (tid == 0) is_last = (atomic_add_acq_rel_gpu(arrivals + u, 1) == n_tiles - 1);
    __syncthreads();
    if (!is_last) return;
  }

  // ---- a3: selection ------------------------------------------------------------
  uint32_t *keys = reinterpret_cast<uint32_t *>(smem);
  uint8_t *flags = reinterpret_cast<uint8_t *>(keys + MB);
  int32_t *cur_sm = reinterpret_cast<int32_t *>(smem + static_cast<size_t>(MB) * 4 + ((MB + 15) & ~15));
  int32_t *prev_sm = cur_sm + MS;
  SelUnit su;
  su.cls = cls;
  su.k = k;
  su.k_e = k_e;
  su.ge = ge;
  su.scores = score_row;
  su.evict = cls == BS_DUAL ? io.evict_logits + static_cast<size_t>(u) * MB : nullptr;
  su.alive = cls == BS_DUAL ? io.alive + static_cast<size_t>(u) * MB : nullptr;
  select_unit_flags<kFrontThreads>(su, keys, flags, sh);
  int total = compact_selection<kFrontThreads>(flags, ge.n_blk, io.cur_idx + srow, MS, cur_sm, sh);
  if (total < 0) {
    if (tid == 0) report(st, BS_ERR_CAPACITY);
    total = 0;
  }
  if (tid == 0) io.cur_cnt[u] = total;

  // ---- a5: set-difference against the previous selection --------------------------
  int np = io.prev_cnt[u];
  if (np < 0 || np > MS) {
    if (tid == 0) report(st, BS_ERR_CAPACITY);
    np = 0;
  }
  for (int i = tid; i < np; i += kFrontThreads) prev_sm[i] = io.prev_idx[srow + i];
  __syncthreads();
  const int na = sorted_diff_into<kFrontThreads>(cur_sm, total, prev_sm, np, io.added + srow, MS, sh);
  const int nr = sorted_diff_into<kFrontThreads>(prev_sm, np, cur_sm, total, io.removed + srow, MS, sh);
  if (tid == 0) {
    io.added_cnt[u] = na;
    io.removed_cnt[u] = nr;
  }

  // ---- a1: the sub-block holding the appended token -------------------------------
  if (tid < 32) {
    const int j = (T - 1) / s;
    const int32_t *pt = kv.page_table + static_cast<size_t>(u) * dims.max_pages_per_unit;
    if (!summary_update_warp<D, KT>(static_cast<const KT *>(kv.k_pool), pt, dims.n_pages, s, T, j,
                                    io.summaries + off + static_cast<int64_t>(j) * D) &&
        tid == 0)
      report(st, BS_ERR_DEVICE_BOUNDS);
  }
  if (tid == 0 && n_tiles > 1) arrivals[u] = 0;  // ready for the next step
}

template <int D, int G>
__global__ void __launch_bounds__(kMmaThreads) step_attn_mma_kernel(bs_dims dims, bs_kv kv, bs_head_cfg cfg,
                                                                    const __grid_constant__ CUtensorMap tmk,
                                                                    const __grid_constant__ CUtensorMap tmv,
                                                                    bs_step_io io, int32_t *arrivals, float *records) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  pdl_launch_dependents();
  attn_split_mma<D, G, true>(dims, io.q, kv, cfg, &tmk, &tmv, io.cur_idx, io.cur_cnt, arrivals, records, io.out,
                             io.lse, io.dev_status, align_smem_1024(smem_raw));
  // Finish only after the selection launch has: work after this step may rely on it.
  pdl_wait();
}

template <int D, int G>
__global__ void __launch_bounds__(kFfmaThreads) step_attn_ffma_kernel(bs_dims dims, bs_kv kv, bs_head_cfg cfg,
                                                                      bs_step_io io, int32_t *arrivals,
                                                                      float *records) {
  extern __shared__ __align__(128) unsigned char smem[];
  pdl_launch_dependents();
  attn_split_ffma<D, G, true>(dims, io.q, kv, cfg, io.cur_idx, io.cur_cnt, arrivals, records, io.out, io.lse,
                              io.dev_status, smem);
  pdl_wait();
}

template <typename K, typename... Args>
cudaError_t launch_pdl(K kernel, dim3 grid, int threads, size_t smem, cudaStream_t cs, Args... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = dim3(threads);
  lc.dynamicSmemBytes = smem;
  lc.stream = cs;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kernel, args...);
}

template <int D, typename KT, int G>
bs_status launch_step(const bs_dims &dims, const bs_kv &kv, const bs_head_cfg &cfg, const bs_step_io &io,
                      int reduce, cudaStream_t cs) {
  constexpr size_t kFrontMaxSmem = 200 * 1024;
  constexpr bool kBf16 = sizeof(KT) == 2;
  constexpr int kAttnSmem = kBf16 ? MmaLayout<D>::kBytes + kSmemAlignSlack : FfmaLayout<D, G>::kBytes;
  static const bool attrs_ok =
      cudaFuncSetAttribute(step_front_kernel<D, KT, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kFrontMaxSmem)) == cudaSuccess &&
      (kBf16 ? cudaFuncSetAttribute(step_attn_mma_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kAttnSmem)
             : cudaFuncSetAttribute(step_attn_ffma_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kAttnSmem)) == cudaSuccess;
  if (!attrs_ok) return BS_ERR_CUDA;
  const int units = dims.batch * dims.n_kv_heads;
  size_t front_smem = front_select_bytes(dims.max_blocks_per_unit, dims.max_sel_per_unit);
  if (front_smem < static_cast<size_t>(ScoreLayout<D, G>::kBytes)) front_smem = ScoreLayout<D, G>::kBytes;
  if (front_smem > kFrontMaxSmem) return BS_ERR_CAPACITY;
  CUtensorMap tk, tv;
  if (kBf16) {
    const bs_status s = make_kv_tensor_maps(dims, kv, &tk, &tv);
    if (s != BS_OK) return s;
  }
  int32_t *counters = static_cast<int32_t *>(io.workspace);
  float *records = static_cast<float *>(io.workspace) + attn_counter_floats(units);
  const dim3 front_grid(dims.max_subs_per_unit / kTileRows + 2, units);
  if (launch_pdl(step_front_kernel<D, KT, G>, front_grid, kFrontThreads, front_smem, cs, dims, kv, cfg, io, reduce,
                 counters) != cudaSuccess)
    return BS_ERR_CUDA;
  const dim3 attn_grid(attn_grid_splits(dims.max_gather_pages_per_unit), units);
  cudaError_t e;
  if (kBf16)
    e = launch_pdl(step_attn_mma_kernel<D, G>, attn_grid, kMmaThreads, static_cast<size_t>(kAttnSmem), cs, dims, kv,
                   cfg, tk, tv, io, counters + units, records);
  else
    e = launch_pdl(step_attn_ffma_kernel<D, G>, attn_grid, kFfmaThreads, static_cast<size_t>(kAttnSmem), cs, dims,
                   kv, cfg, io, counters + units, records);
  return e == cudaSuccess ? BS_OK : BS_ERR_CUDA;
}

template <int D, typename KT>
bs_status dispatch_g(int G, const bs_dims &dims, const bs_kv &kv, const bs_head_cfg &cfg, const bs_step_io &io,
                     int reduce, cudaStream_t cs) {
  switch (G) {
    case 1: return launch_step<D, KT, 1>(dims, kv, cfg, io, reduce, cs);
    case 2: return launch_step<D, KT, 2>(dims, kv, cfg, io, reduce, cs);
    case 3: return launch_step<D, KT, 3>(dims, kv, cfg, io, reduce, cs);
    case 4: return launch_step<D, KT, 4>(dims, kv, cfg, io, reduce, cs);
    case 5: return launch_step<D, KT, 5>(dims, kv, cfg, io, reduce, cs);
    case 6: return launch_step<D, KT, 6>(dims, kv, cfg, io, reduce, cs);
    case 7: return launch_step<D, KT, 7>(dims, kv, cfg, io, reduce, cs);
    default: return launch_step<D, KT, 8>(dims, kv, cfg, io, reduce, cs);
  }
}

}  // namespace
}  // namespace bsi

extern "C" bs_status bs_decode_step(const bs_dims *dims, const bs_kv *kv, const bs_head_cfg *cfg,
                                    const bs_step_io *io, bs_group_reduce group_reduce, bs_stream_t stream) {
  using namespace bsi;
  bs_status s = check_dims(dims);
  if (s != BS_OK) return s;
  if (!kv || !cfg || !io || !kv->k_pool || !kv->v_pool || !kv->page_table || !kv->seq_lens || !cfg->cls ||
      !cfg->block_tokens || !cfg->sub_tokens || !cfg->k_total || !cfg->k_evict || !cfg->sink_tokens ||
      !cfg->local_tokens || !cfg->sum_off || !cfg->sum_rows || !io->q || !io->summaries || !io->scores ||
      !io->prev_idx || !io->prev_cnt || !io->cur_idx || !io->cur_cnt || !io->added || !io->added_cnt ||
      !io->removed || !io->removed_cnt || !io->out || !io->lse || !io->workspace || !io->dev_status)
    return BS_ERR_INVALID_ARG;
  if (group_reduce != BS_GROUP_MAX && group_reduce != BS_GROUP_MEAN) return BS_ERR_INVALID_ARG;
  if (io->prev_idx == io->cur_idx || io->prev_cnt == io->cur_cnt) return BS_ERR_INVALID_ARG;
  if (!aligned16(io->q) || !aligned16(kv->k_pool) || !aligned16(kv->v_pool) || !aligned16(io->out) ||
      !aligned16(io->workspace) || !aligned16(io->summaries))
    return BS_ERR_ALIGN;
  if (io->workspace_bytes < bs_workspace_size(dims)) return BS_ERR_CAPACITY;
  if (dims->max_sel_per_unit > kStepMaxSel) return BS_ERR_CAPACITY;
  const int G = dims->n_q_heads / dims->n_kv_heads;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (dims->head_dim == 128) {
    if (dims->kv_dtype == BS_BF16) return dispatch_g<128, uint16_t>(G, *dims, *kv, *cfg, *io, group_reduce, cs);
    return dispatch_g<128, float>(G, *dims, *kv, *cfg, *io, group_reduce, cs);
  }
  if (dims->kv_dtype == BS_BF16) return dispatch_g<64, uint16_t>(G, *dims, *kv, *cfg, *io, group_reduce, cs);
  return dispatch_g<64, float>(G, *dims, *kv, *cfg, *io, group_reduce, cs);
}
