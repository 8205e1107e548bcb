// Set-difference-driven block swap into a GPU block cache: "Technisches Resümee: NOSA",
// Methodik / 2. System: NOSI (KV cache in minimal block units; set-difference kernels
// for block swapping; host-to-device transfer kernels over Unified Virtual
// Addressing) and Lokalitätsgarantie (blocks kept between steps stay in the GPU cache).
//
// Launch 1, swap_book_kernel (one CTA per unit): frees the slots of the removed
// blocks, lists the free slots in ascending order (one ordered compaction), gives them
// to the added blocks in order and rewrites the cache page table.
// Launch 2, swap_copy_kernel (one CTA per (added block, unit), plus one per unit for
// the page holding the appended token T-1 when its block stays cached): copies pages,
// K and V, from host memory into the block's slot with 16-byte loads issued eight at
// a time per thread before their stores.
#include "bs_select_impl.cuh"

namespace bsi {
namespace {

constexpr int kSwapThreads = 256;
constexpr int kCopyThreads = 128;
constexpr int kMaxSlots = 4096;

__device__ __forceinline__ int64_t slot_page(int u, int slots, int s, int pps, int p) {
  return (static_cast<int64_t>(u) * slots + s) * pps + p;
}

__global__ void __launch_bounds__(kSwapThreads) swap_book_kernel(bs_dims dims, bs_head_cfg cfg,
                                                                 const int32_t *__restrict__ seq_lens,
                                                                 bs_block_cache cache, const int32_t *__restrict__ added,
                                                                 const int32_t *__restrict__ added_cnt,
                                                                 const int32_t *__restrict__ removed,
                                                                 const int32_t *__restrict__ removed_cnt, int32_t *st) {
  __shared__ SelShared<kSwapThreads> sh;
  __shared__ int16_t free_sm[kMaxSlots];
  const int u = blockIdx.x, tid = threadIdx.x;
  const int b = u / dims.n_kv_heads;
  const int MB = dims.max_blocks_per_unit, MS = dims.max_sel_per_unit, MP = dims.max_pages_per_unit;
  const int S = cache.slots_per_unit, PPS = cache.pages_per_slot;
  const int g = cfg.block_tokens[u];
  const int T = seq_lens[b];
  if (g <= 0 || g % kPage != 0 || g / kPage > PPS || T < 1) {
    if (tid == 0) report(st, BS_ERR_INVALID_ARG);
    return;
  }
  const int ppb = g / kPage;
  int32_t *sb = cache.slot_block + static_cast<size_t>(u) * S;
  int32_t *bsl = cache.block_slot + static_cast<size_t>(u) * MB;
  int32_t *pt = cache.page_table + static_cast<size_t>(u) * MP;
  int nr = removed_cnt[u], na = added_cnt[u];
  if (nr < 0 || nr > MS || na < 0 || na > MS) {
    if (tid == 0) report(st, BS_ERR_CAPACITY);
    nr = max(0, min(nr, MS));
    na = max(0, min(na, MS));
  }
  // 1. removed blocks leave the cache
  for (int i = tid; i < nr; i += kSwapThreads) {
    const int c = removed[static_cast<size_t>(u) * MS + i];
    if (c < 0 || c >= MB) {
      report(st, BS_ERR_DEVICE_BOUNDS);
      continue;
    }
    const int s = bsl[c];
    if (s >= 0 && s < S) sb[s] = -1;
    bsl[c] = -1;
    for (int p = 0; p < ppb; ++p) {
      const int lp = c * ppb + p;
      if (lp < MP) pt[lp] = -1;
    }
  }
  __syncthreads();
  // 2. free slots, ascending
  const int per = (S + kSwapThreads - 1) / kSwapThreads;
  const int a = tid * per, e = min(S, a + per);
  int mine = 0;
  for (int s = a; s < e; ++s) mine += sb[s] < 0 ? 1 : 0;
  int n_free;
  int pos = block_excl_scan<kSwapThreads>(mine, sh, &n_free);
  for (int s = a; s < e; ++s)
    if (sb[s] < 0) free_sm[pos++] = static_cast<int16_t>(s);
  __syncthreads();
  // 3. added blocks take the free slots in order
  for (int i = tid; i < na; i += kSwapThreads) {
    const int c = added[static_cast<size_t>(u) * MS + i];
    if (c < 0 || c >= MB) {
      report(st, BS_ERR_DEVICE_BOUNDS);
      continue;
    }
    if (i >= n_free) {
      report(st, BS_ERR_CAPACITY);
      continue;
    }
    const int s = free_sm[i];
    sb[s] = c;
    bsl[c] = s;
    for (int p = 0; p < ppb; ++p) {
      const int lp = c * ppb + p;
      if (lp < MP) pt[lp] = lp * kPage < T ? static_cast<int32_t>(slot_page(u, S, s, PPS, p)) : -1;
    }
  }
  __syncthreads();
  // 4. the tail block (it holds token T-1) may have grown a page since it was cached
  if (tid == 0) {
    const int c = (T - 1) / g;
    const int s = c < MB ? bsl[c] : -1;
    const int lp = (T - 1) / kPage;
    if (s >= 0 && lp < MP) pt[lp] = static_cast<int32_t>(slot_page(u, S, s, PPS, lp - c * ppb));
  }
}

__global__ void __launch_bounds__(kCopyThreads) swap_copy_kernel(bs_dims dims, bs_head_cfg cfg,
                                                                 const int32_t *__restrict__ seq_lens, bs_host_kv host,
                                                                 bs_block_cache cache, const int32_t *__restrict__ added,
                                                                 const int32_t *__restrict__ added_cnt, int32_t *st) {
  const int i = blockIdx.x, u = blockIdx.y, tid = threadIdx.x;
  const int MS = dims.max_sel_per_unit, MB = dims.max_blocks_per_unit, MP = dims.max_pages_per_unit;
  const int g = cfg.block_tokens[u];
  const int T = seq_lens[u / dims.n_kv_heads];
  if (g <= 0 || g % kPage != 0 || T < 1) return;  // reported by the bookkeeping
  const int ppb = g / kPage;
  const int na = min(added_cnt[u], MS);
  int c, p0, np;
  if (i < MS) {
    // CTA i < MS: added block i, every page of it that holds tokens
    if (i >= na) return;
    c = added[static_cast<size_t>(u) * MS + i];
    p0 = 0;
    np = 0;
    while (c >= 0 && np < ppb && (c * ppb + np) * kPage < T && c * ppb + np < MP) ++np;
  } else {
    // CTA MS: the page holding token T-1 (the appended token) when its block was cached
    // earlier (an added block's pages are copied above)
    c = (T - 1) / g;
    for (int j = 0; j < na; ++j)
      if (added[static_cast<size_t>(u) * MS + j] == c) return;
    p0 = (T - 1) / kPage - c * ppb;
    np = 1;
  }
  if (c < 0 || c >= MB) return;  // reported by the bookkeeping
  const int s = cache.block_slot[static_cast<size_t>(u) * MB + c];
  if (s < 0) return;  // not cached (or not placed: capacity, reported)
  const int S = cache.slots_per_unit, PPS = cache.pages_per_slot;
  const int esz = dims.kv_dtype == BS_BF16 ? 2 : 4;
  const int vec_per_page = kPage * dims.head_dim * esz / 16;
  const int total = np * 2 * vec_per_page;  // K then V of each page
  const int32_t *hpt = host.page_table + static_cast<size_t>(u) * MP + static_cast<size_t>(c) * ppb + p0;
  constexpr int kBatch = 8;
  for (int base = tid; base < total; base += kCopyThreads * kBatch) {
    uint4 v[kBatch];
    const uint4 *src[kBatch];
    uint4 *dst[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      src[j] = nullptr;
      dst[j] = nullptr;
      const int idx = base + j * kCopyThreads;
      if (idx < total) {
        const int p = idx / (2 * vec_per_page);
        const int r = idx - p * 2 * vec_per_page;
        const int pool = r / vec_per_page, w = r - pool * vec_per_page;
        const int hp = hpt[p];
        if (hp < 0 || hp >= host.n_pages) {
          report(st, BS_ERR_DEVICE_BOUNDS);
          continue;
        }
        const size_t page_vecs = static_cast<size_t>(vec_per_page);
        const uint4 *hbase = static_cast<const uint4 *>(pool == 0 ? host.k_pool : host.v_pool);
        uint4 *dbase = static_cast<uint4 *>(pool == 0 ? cache.k_pool : cache.v_pool);
        src[j] = hbase + static_cast<size_t>(hp) * page_vecs + w;
        dst[j] = dbase + static_cast<size_t>(slot_page(u, S, s, PPS, p0 + p)) * page_vecs + w;
      }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      if (src[j]) v[j] = *src[j];
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      if (dst[j]) *dst[j] = v[j];
  }
}

}  // namespace
}  // namespace bsi

extern "C" bs_status bs_block_swap(const bs_dims *dims, const bs_head_cfg *cfg, const int32_t *seq_lens,
                                   const bs_host_kv *host, const bs_block_cache *cache, const int32_t *added,
                                   const int32_t *added_cnt, const int32_t *removed, const int32_t *removed_cnt,
                                   int32_t *dev_status, bs_stream_t stream) {
  using namespace bsi;
  bs_status s = check_dims(dims);
  if (s != BS_OK) return s;
  if (!cfg || !cfg->block_tokens || !seq_lens || !host || !cache || !added || !added_cnt || !removed ||
      !removed_cnt || !dev_status || !host->k_pool || !host->v_pool || !host->page_table || !cache->k_pool ||
      !cache->v_pool || !cache->page_table || !cache->slot_block || !cache->block_slot)
    return BS_ERR_INVALID_ARG;
  if (cache->slots_per_unit < 1 || cache->slots_per_unit > kMaxSlots || cache->pages_per_slot < 1 ||
      host->n_pages < 1)
    return BS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(host->k_pool) | reinterpret_cast<uintptr_t>(host->v_pool) |
       reinterpret_cast<uintptr_t>(cache->k_pool) | reinterpret_cast<uintptr_t>(cache->v_pool)) & 15u)
    return BS_ERR_ALIGN;
  const int units = dims->batch * dims->n_kv_heads;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  swap_book_kernel<<<units, kSwapThreads, 0, cs>>>(*dims, *cfg, seq_lens, *cache, added, added_cnt, removed,
                                                   removed_cnt, dev_status);
  if (cudaGetLastError() != cudaSuccess) return BS_ERR_CUDA;
  swap_copy_kernel<<<dim3(dims->max_sel_per_unit + 1, units), kCopyThreads, 0, cs>>>(*dims, *cfg, seq_lens, *host,
                                                                                 *cache, added, added_cnt,
                                                                                 dev_status);
  return launch_status();
}
