// a3: per-unit block selection.
// Streaming vs retrieval heads: "Technische Samenvatting: Fluxion", Kerninzichten
// item 2; dual selection with the strict eviction rule and selection on
// pre-exponential logits: "Technisches Resümee: NOSA", Methodik / 1. Algorithmus:
// NOSA, "Dual-Selection-Mechanismus" and "ED-DMA".
//
// One CTA per unit. Keys are float32 values mapped to order-preserving uint32. The
// k-th largest key is found by a four-pass 8-bit radix select (histograms in shared
// memory, warp-aggregated with __match_any_sync); every key above it is taken, and of
// the keys equal to it the lowest block indices are taken (a block-wide prefix count
// in index order). The final set is written in ascending order by a compaction over
// block indices, so no sort is needed.
#include "bs_internal.cuh"

namespace bsi {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;

// flag bits per block
constexpr uint8_t kSel = 1;     // in the final selection
constexpr uint8_t kAlive = 2;   // eligible for Gamma_e (dual)
constexpr uint8_t kEvict = 4;   // chosen by Gamma_e
constexpr uint8_t kElig = 8;    // eligible in the current top-k pass

struct SelShared {
  uint32_t hist[256];
  int warp_tot[kSelWarps];
  int bcast[4];
};

// Exclusive prefix sum of one int per thread over the CTA; *total gets the sum.
__device__ __forceinline__ int block_excl_scan(int v, SelShared &sh, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh.warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kSelWarps ? sh.warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kSelWarps) sh.warp_tot[lane] = w;  // inclusive
  }
  __syncthreads();
  const int before = (warp > 0 ? sh.warp_tot[warp - 1] : 0) + x - v;
  *total = sh.warp_tot[kSelWarps - 1];
  __syncthreads();
  return before;
}

// Marks with `mark` the k blocks of [lo, hi) carrying kElig with the largest keys,
// lower index first among equal keys.
__device__ void topk_mark(const uint32_t *keys, uint8_t *flags, int lo, int hi, int k, uint8_t mark,
                          SelShared &sh) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int n = hi - lo;
  if (k <= 0 || n <= 0) return;
  // Contiguous per-thread ranges keep the index order for the tie pass.
  const int per = (n + kSelThreads - 1) / kSelThreads;
  const int a = lo + tid * per, e = min(hi, a + per);
  int my = 0;
  for (int c = a; c < e; ++c) my += (flags[c] & kElig) ? 1 : 0;
  int n_elig;
  block_excl_scan(my, sh, &n_elig);
  if (k >= n_elig) {
    for (int c = a; c < e; ++c)
      if (flags[c] & kElig) flags[c] |= mark;
    __syncthreads();
    return;
  }
  uint32_t prefix = 0, pmask = 0;
  int rem = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kSelThreads) sh.hist[i] = 0;
    __syncthreads();
    for (int base = lo; base < hi; base += kSelThreads) {
      const int c = base + tid;
      bool valid = false;
      uint32_t digit = 256;
      if (c < hi && (flags[c] & kElig)) {
        const uint32_t key = keys[c - lo];
        if ((key & pmask) == prefix) {
          valid = true;
          digit = (key >> shift) & 255u;
        }
      }
      const unsigned peers = __match_any_sync(0xffffffffu, digit);
      if (valid && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[digit], static_cast<uint32_t>(__popc(peers)));
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns bins [255-8l-7, 255-8l], scanned from the top.
      int cnt = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) cnt += static_cast<int>(sh.hist[255 - 8 * lane - i]);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int before = incl - cnt;
      if (before < rem && rem <= incl) {
        int run = before;
        for (int i = 0; i < 8; ++i) {
          const int bin = 255 - 8 * lane - i;
          const int h = static_cast<int>(sh.hist[bin]);
          if (run + h >= rem) {
            sh.bcast[0] = bin;
            sh.bcast[1] = rem - run;
            break;
          }
          run += h;
        }
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(sh.bcast[0]) << shift;
    pmask |= 255u << shift;
    rem = sh.bcast[1];
    __syncthreads();
  }
  // prefix is the k-th largest key; `rem` of the keys equal to it are taken.
  int eq = 0;
  for (int c = a; c < e; ++c) {
    if (!(flags[c] & kElig)) continue;
    const uint32_t key = keys[c - lo];
    if (key > prefix) flags[c] |= mark;
    else if (key == prefix) ++eq;
  }
  int tot;
  int rank = block_excl_scan(eq, sh, &tot);
  for (int c = a; c < e; ++c) {
    if (!(flags[c] & kElig) || keys[c - lo] != prefix) continue;
    if (rank < rem) flags[c] |= mark;
    ++rank;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(bs_dims dims, bs_head_cfg cfg,
                                                             const int32_t *__restrict__ seq_lens,
                                                             const float *__restrict__ scores,
                                                             const float *__restrict__ evict, uint8_t *alive,
                                                             int32_t *__restrict__ sel_idx,
                                                             int32_t *__restrict__ sel_cnt, int32_t *st) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ SelShared sh;
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
  const Geom ge = unit_geom(T, g, s, cfg.sink_tokens[u], cfg.local_tokens[u]);
  const int lo = ge.c_lo, hi = ge.c_hi;
  const size_t row = static_cast<size_t>(u) * MB;

  // Forced blocks; candidates [lo, hi) start unflagged.
  for (int c = tid; c < ge.n_blk; c += kSelThreads) {
    const bool forced = c < ge.n_sink || c >= ge.local_lo;
    uint8_t f = forced ? kSel : 0;
    if (cls == BS_DUAL && c >= lo && c < hi && alive[row + c]) f |= kAlive;
    flags[c] = f;
  }
  __syncthreads();

  if (cls == BS_RETRIEVAL) {
    for (int c = lo + tid; c < hi; c += kSelThreads) {
      keys[c - lo] = order_key(scores[row + c]);
      flags[c] |= kElig;
    }
    __syncthreads();
    topk_mark(keys, flags, lo, hi, k, kSel, sh);
  } else if (cls == BS_DUAL) {
    // Gamma_e: the k_e largest eviction logits among alive candidates.
    for (int c = lo + tid; c < hi; c += kSelThreads) {
      keys[c - lo] = order_key(evict[row + c]);
      if (flags[c] & kAlive) flags[c] |= kElig;
    }
    __syncthreads();
    topk_mark(keys, flags, lo, hi, k_e, kEvict, sh);
    // Strict eviction: candidates outside Gamma_e are dead from now on. Gamma_q: the
    // k - k_e largest scores among the candidates outside Gamma_e.
    for (int c = lo + tid; c < hi; c += kSelThreads) {
      const uint8_t f = flags[c];
      alive[row + c] = (f & kEvict) ? 1 : 0;
      keys[c - lo] = order_key(scores[row + c]);
      flags[c] = static_cast<uint8_t>(((f & kEvict) ? kSel : kElig) | (f & kEvict));
    }
    __syncthreads();
    topk_mark(keys, flags, lo, hi, k - k_e, kSel, sh);
  }

  // Ascending compaction of the selected blocks.
  const int per = (ge.n_blk + kSelThreads - 1) / kSelThreads;
  const int a = tid * per, e = min(ge.n_blk, a + per);
  int mine = 0;
  for (int c = a; c < e; ++c) mine += (flags[c] & kSel) ? 1 : 0;
  int total;
  int pos = block_excl_scan(mine, sh, &total);
  if (total > dims.max_sel_per_unit) {
    if (tid == 0) {
      report(st, BS_ERR_CAPACITY);
      sel_cnt[u] = 0;
    }
    for (int i = tid; i < dims.max_sel_per_unit; i += kSelThreads) out[i] = -1;
    return;
  }
  for (int c = a; c < e; ++c)
    if (flags[c] & kSel) out[pos++] = c;
  for (int i = total + tid; i < dims.max_sel_per_unit; i += kSelThreads) out[i] = -1;
  if (tid == 0) sel_cnt[u] = total;
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
