// The fused decode step of one layer: all five steps of the path in two launches.
//
// Launch 1, step_front_kernel, one CTA per (unit, group of score tiles), unit-fastest:
//   * the CTAs of a retrieval or dual unit score its candidate blocks (a2), one or
//     several 64-row tiles each; the unit's first CTA also recomputes the sub-block
//     holding the token just appended (a1). That sub-block lies in the always-forced
//     tail block, which no score of this step reads, so a1 runs beside a2;
//   * the last CTA of each unit to finish (an integer arrival ticket, one acquire-
//     release atomic per CTA) selects the unit's blocks (a3), writes the page list of
//     the selection for the attention, publishes the selection (its count is written
//     last, with a release store) and writes its set-difference against the previous
//     step (a5);
//   * a streaming unit has one CTA that does a1, a3 and a5.
// Launch 2, the attention (a4) as a programmatic dependent launch: streaming units'
// splits need no selection and start while launch 1 is still working; every other
// unit's splits wait (bounded) until their unit's selection count is published.
//
// Both kernels are programmatic dependents of the work before them in the stream: they
// read only the per-unit head configuration before waiting for it to finish.
#include <algorithm>

#include "bs_attn_launch.cuh"
#include "bs_score_impl.cuh"
#include "bs_select_impl.cuh"
#include "bs_summaries_impl.cuh"

namespace bsi {
namespace {

constexpr int kFrontThreads = 256;
constexpr int kStepMaxSel = 4096;

__device__ __forceinline__ void pdl_wait_front() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger_front() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void store_release(int32_t *p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Publishes unit u's selection count for the attention: (epoch << 16) | count with a
// release store, the epoch one past the one the attention last took (expect[u]; read
// after the previous step's attention has finished, and written only by that attention
// once every reader of the unit's word is done). A count that is not this step's cannot
// match, whatever the timing.
__device__ __forceinline__ void publish_selection(const StepWords &w, int u, int count) {
  const int e = (__ldcg(w.expect + u) + 1) & kEpochMask;
  store_release(w.pub + u, (e << 16) | count);
}
__device__ __forceinline__ int ticket_acq_rel(int32_t *p) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
  return old;
}

// Exclusive prefix sum of one int per thread over the CTA (kFrontThreads threads) via
// shared tmp (one int per warp); *total gets the sum. All threads call it.
__device__ __forceinline__ int front_scan(int v, int *tmp, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kFrontThreads / 32; ++w) {
    const int t = tmp[w];
    if (w < warp) before += t;
    tot += t;
  }
  __syncthreads();
  *total = tot;
  return before + x - v;
}

// The rank k whose items [pos[k], pos[k + 1]) hold item p (pos ascending, pos[U] = W;
// U when p >= W).
__device__ __forceinline__ int stream_rank_at(const int *pos, int U, int p) {
  int lo = 0, hi = U;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (pos[mid + 1] <= p) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Shared memory of the selection phase: keys [MB] u32 and flags [MB] u8 (padded to
// 16; used by selections above 32 candidates per thread), current and previous
// selection [MS] i32 each, then (page lists in cluster mode, tables up to 64 KB) the
// unit's page-table row [max_pages] i32.
constexpr int kPtCacheInts = 16384;
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__host__ __device__ inline size_t front_select_bytes(int max_blocks, int max_sel, int pt_cache_ints) {
  const size_t flags = (static_cast<size_t>(max_blocks) + 15) & ~size_t(15);
  return static_cast<size_t>(max_blocks) * 4 + flags + 2 * static_cast<size_t>(max_sel) * 4 +
         (pt_cache_ints > 0 ? static_cast<size_t>(pt_cache_ints) * 4 + 32 : 0);
}

// ---------------------------------------------------------------------------
// The per-unit end of the front kernels, all NT threads of the CTA: selection (a3), the
// page list of the selection for the attention, the published count, and the
// set-difference against the previous selection (a5). `smem` is the CTA's dynamic
// shared memory (at least front_select_bytes(MB, MS, pt_cache_ints) bytes, no copy in
// flight into it). The unit's scores (retrieval and dual units) are complete.
// ---------------------------------------------------------------------------
struct UnitFront {
  int u, cls, k, k_e, g, T;
  Geom ge;
};

template <int NT>
__device__ __forceinline__ void unit_select_publish(const bs_dims &dims, const bs_kv &kv, const bs_step_io &io,
                                                 const StepWords &words, int32_t *plist, int pt_cache_ints,
                                                 unsigned char *smem, SelShared<NT> &sh, const UnitFront &uf) {
  const int tid = threadIdx.x;
  const int MB = dims.max_blocks_per_unit, MS = dims.max_sel_per_unit;
  const int u = uf.u, cls = uf.cls, k = uf.k, k_e = uf.k_e, g = uf.g, T = uf.T;
  const Geom &ge = uf.ge;
  int32_t *st = io.dev_status;
  const size_t srow = static_cast<size_t>(u) * MS;
  float *score_row = io.scores + static_cast<size_t>(u) * MB;
  // ---- a3: selection ------------------------------------------------------------
  uint32_t *keys = reinterpret_cast<uint32_t *>(smem);
  uint8_t *flags = reinterpret_cast<uint8_t *>(keys + MB);
  int32_t *cur_sm = reinterpret_cast<int32_t *>(smem + static_cast<size_t>(MB) * 4 + ((MB + 15) & ~15));
  int32_t *prev_sm = cur_sm + MS;
  int32_t *pt_sm = reinterpret_cast<int32_t *>((reinterpret_cast<uintptr_t>(prev_sm + MS) + 15) & ~uintptr_t(15));
  // The previous selection is final since the previous step: copy it asynchronously
  // (cp.async) into shared memory; it lands while the selection runs. So does the
  // unit's page-table row when the page list is written from shared memory: one bulk
  // copy of its 16-byte-aligned span (starting up to three entries early, inside the
  // table), the last few entries past that span read directly.
  __shared__ int np_sm;
  __shared__ uint64_t pt_bar;
  if (tid == 0) cp_async4(&np_sm, io.prev_cnt + u);
  for (int i = tid; i < MS; i += NT) cp_async4(prev_sm + i, io.prev_idx + srow + i);
  cp_async_commit();
  const bool mk_plist = plist != nullptr && cls != BS_STREAMING;
  const int32_t *pt_row = kv.page_table + static_cast<size_t>(u) * dims.max_pages_per_unit;
  const int n_lp = min(dims.max_pages_per_unit, (T + kPage - 1) / kPage);
  const uintptr_t pt_a = reinterpret_cast<uintptr_t>(pt_row);
  const uintptr_t pt_a0 = pt_a & ~uintptr_t(15);
  const uintptr_t pt_e0 = (pt_a + static_cast<uintptr_t>(n_lp) * 4) & ~uintptr_t(15);
  const bool pt_cached = mk_plist && pt_cache_ints >= n_lp && pt_e0 > pt_a0;
  const int pt_lead = static_cast<int>((pt_a - pt_a0) / 4);             // entries before the row
  int pt_in_smem = pt_cached ? static_cast<int>((pt_e0 - pt_a) / 4) : 0;  // row entries copied
  if (pt_cached && tid == 0) {
    mbar_init(&pt_bar, 1);
    fence_mbar_init();
    const uint32_t bytes = static_cast<uint32_t>(pt_e0 - pt_a0);
    mbar_arrive_expect_tx(&pt_bar, bytes);
    bulk_g2s(pt_sm, reinterpret_cast<const void *>(pt_a0), bytes, &pt_bar);
  }
  SelUnit su;
  su.cls = cls;
  su.k = k;
  su.k_e = k_e;
  su.ge = ge;
  su.scores = score_row;
  su.evict = cls == BS_DUAL ? io.evict_logits + static_cast<size_t>(u) * MB : nullptr;
  su.alive = cls == BS_DUAL ? io.alive + static_cast<size_t>(u) * MB : nullptr;
  int total = select_unit<NT>(su, keys, flags, io.cur_idx + srow, MS, cur_sm, sh);
  if (total < 0) {
    if (tid == 0) report(st, BS_ERR_CAPACITY);
    total = 0;
  }
  if (mk_plist) {
    // Page list for the attention: the pages of the selected blocks in order (the
    // last selected block is the tail block; its pages past T are left out), -1 for
    // an entry outside the table or the pool.
    __syncthreads();
    if (pt_cached && !mbar_wait_bounded(&pt_bar, 0, st)) pt_in_smem = 0;  // (reported) read global instead
    __syncthreads();
    const int ppb = g / kPage;
    const int tail_pages = min(ppb, (T - (ge.n_blk - 1) * g + kPage - 1) / kPage);
    const int n_pages = total > 0 ? (total - 1) * ppb + tail_pages : 0;
    int32_t *pl = plist + static_cast<size_t>(u) * dims.max_gather_pages_per_unit;
    if (n_pages <= dims.max_gather_pages_per_unit) {
      // Four entries a thread per round, their page-table loads issued before any store.
      constexpr int kB = 4;
      for (int i0 = tid; i0 < n_pages; i0 += NT * kB) {
        int phys[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          const int i = i0 + j * NT;
          phys[j] = -1;
          if (i < n_pages) {
            const int blk = i / ppb, pb = i - blk * ppb;
            const int c = cur_sm[blk];
            const int lp = c * ppb + pb;
            if (c >= 0 && lp < n_lp && c * g + pb * kPage < T)
              phys[j] = lp < pt_in_smem ? pt_sm[pt_lead + lp] : __ldg(pt_row + lp);
          }
        }
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          const int i = i0 + j * NT;
          if (i < n_pages) pl[i] = (phys[j] < 0 || phys[j] >= dims.n_pages) ? -1 : phys[j];
        }
      }
    }
  }
  // Publish: the row and the page list are written; the count (release) tells the
  // attention they are ready.
  __syncthreads();
  if (tid == 0) {
    io.cur_cnt[u] = total;
    publish_selection(words, u, total);
  }
  cp_async_wait_all();
  __syncthreads();
  int np = np_sm;
  if (np < 0 || np > MS) {
    if (tid == 0) report(st, BS_ERR_CAPACITY);
    np = 0;
  }

  // ---- a5: set-difference against the previous selection --------------------------
  const int2 nd = setdiff_sorted<NT>(cur_sm, total, prev_sm, np, io.added + srow, io.removed + srow, MS, sh);
  if (tid == 0) {
    io.added_cnt[u] = nd.x;
    io.removed_cnt[u] = nd.y;
  }
}

// A unit whose configuration or length breaks a rule: an empty selection (row -1,
// counts 0) published as such, the code reported. All threads of the CTA.
__device__ __forceinline__ void unit_error_publish(const bs_dims &dims, const bs_step_io &io, const StepWords &words,
                                                int u, int code) {
  const int tid = threadIdx.x, MS = dims.max_sel_per_unit;
  const size_t srow = static_cast<size_t>(u) * MS;
  for (int i = tid; i < MS; i += blockDim.x) io.cur_idx[srow + i] = io.added[srow + i] = io.removed[srow + i] = -1;
  __syncthreads();
  if (tid == 0) {
    report(io.dev_status, code);
    io.added_cnt[u] = 0;
    io.removed_cnt[u] = 0;
    io.cur_cnt[u] = 0;
    publish_selection(words, u, 0);
  }
}

// a1 for unit u: the sub-block holding token T-1 (one warp: call with the 32 lanes of
// one warp only).
template <int D>
__device__ __forceinline__ void unit_summary_update(const bs_dims &dims, const bs_kv &kv, const bs_step_io &io,
                                                    int u, int s, int T, int64_t sum_off, int32_t *st) {
  const int j = (T - 1) / s;
  const int32_t *pt = kv.page_table + static_cast<size_t>(u) * dims.max_pages_per_unit;
  float *row = io.summaries + sum_off + static_cast<int64_t>(j) * D;
  const bool ok = dims.kv_dtype == BS_BF16
                      ? summary_update_warp<D, uint16_t>(static_cast<const uint16_t *>(kv.k_pool), pt, dims.n_pages,
                                                         s, T, j, row)
                      : summary_update_warp<D, float>(static_cast<const float *>(kv.k_pool), pt, dims.n_pages, s, T,
                                                      j, row);
  if (!ok && (threadIdx.x & 31) == 0) report(st, BS_ERR_DEVICE_BOUNDS);
}

template <int D, int G>
__global__ void __launch_bounds__(kFrontThreads, 2) step_front_kernel(bs_dims dims, bs_kv kv, bs_head_cfg cfg,
                                                                   bs_step_io io, int reduce, StepWords words,
                                                                   int32_t *plist, int pt_cache_ints, int tpc) {
  using L = ScoreLayout<D, G>;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t bars[2];
  __shared__ SelShared<kFrontThreads> sh;
  __shared__ int is_last;
  // CTA j of unit u scores tiles [j * tpc, (j + 1) * tpc); grid is unit-fastest so every
  // unit's first CTA comes first.
  const int u = blockIdx.x, cj = blockIdx.y, tid = threadIdx.x;
  const int b = u / dims.n_kv_heads, hk = u % dims.n_kv_heads;
  const int MB = dims.max_blocks_per_unit, MS = dims.max_sel_per_unit;
  const int nbuf = tpc > 1 ? 2 : 1;
  int32_t *st = io.dev_status;
  // Per-unit head configuration: read before the preceding work has finished.
  const int cls = cfg.cls[u], g = cfg.block_tokens[u], s = cfg.sub_tokens[u];
  const int k = cfg.k_total[u], k_e = cfg.k_evict[u], sink = cfg.sink_tokens[u], local = cfg.local_tokens[u];
  const int64_t off = cfg.sum_off[u];
  const int rows = cfg.sum_rows[u];
  const bool cfg_ok = unit_cfg_ok(cls, g, s, k, k_e, sink, local);
  const bool scored = cfg_ok && cls != BS_STREAMING;
  // First summary row of tile t: candidates start after the sink blocks (the checks
  // below confirm this once the length is known; otherwise the unit has no candidates).
  const int64_t row_base = scored ? static_cast<int64_t>((sink + g - 1) / g) * (g / s) : -1;
  auto tile_row = [&](int t) -> int64_t { return scored ? row_base + static_cast<int64_t>(t) * kTileRows : -1; };
  const int t0 = cj * tpc;
  // CTAs past every tile the unit can have leave before waiting.
  if (cj > 0 && (!scored || tile_row(t0) >= rows)) return;
  pdl_wait_front();  // q, lengths, KV pages, summaries and selection state are now final
  int32_t *arrivals = words.tickets;
  score_bars_init(bars, nbuf);
  __syncthreads();
  pdl_trigger_front();  // the attention may start launching
  // A CTA starts the copies of its first tiles before reading the length when it takes
  // one tile (short, latency-bound launches) or is its unit's first; the later CTAs of
  // multi-tile launches read it first and copy only rows of the unit's candidates (with
  // unequal lengths in a batch, their tiles often lie past them). Every path below waits
  // for whatever is in flight (drain) before returning or reusing memory.
  const bool spec = scored && off >= 0 && off % 4 == 0;
  const float *summ = io.summaries + (spec ? off : 0);
  int64_t first_end = rows;
  if (cj > 0 && tpc > 1 && spec) {
    const int T0 = kv.seq_lens[b];
    if (T0 >= 1) {
      const int64_t cand_end = static_cast<int64_t>(unit_geom(T0, g, s, sink, local).c_hi) * (g / s);
      first_end = min(static_cast<int64_t>(rows), cand_end);
    }
  }
  int inflight[2] = {0, 0}, uses[2] = {0, 0};
  for (int i = 0; i < nbuf && i < tpc; ++i)
    inflight[i] = score_copy<D>(summ, spec ? tile_row(t0 + i) : -1, first_end, smem + i * L::kTileBytes, &bars[i]);
  // The queries too: their loads fly beside the copies and the length's.
  const size_t qbase = (static_cast<size_t>(b) * dims.n_q_heads + static_cast<size_t>(hk) * G) * D;
  const void *qrow = dims.q_dtype == BS_BF16
                         ? static_cast<const void *>(static_cast<const uint16_t *>(io.q) + qbase)
                         : static_cast<const void *>(static_cast<const float *>(io.q) + qbase);
  float *qs = reinterpret_cast<float *>(smem + L::off_q(nbuf));
  if (scored) score_load_q<D, G>(qs, qrow, dims.q_dtype);
  auto wait_buf = [&](int i) -> bool {
    const bool ok = score_wait(&bars[i], static_cast<uint32_t>(uses[i] & 1), inflight[i], st);
    if (inflight[i] > 0) ++uses[i];
    inflight[i] = 0;
    return ok;
  };
  auto drain = [&]() -> bool {
    bool ok = true;
    for (int i = 0; i < nbuf; ++i) ok = wait_buf(i) && ok;
    return ok;
  };

  const int T = kv.seq_lens[b];
  int code = BS_OK;
  if (!cfg_ok || T < 1) code = BS_ERR_INVALID_ARG;
  else if (cls == BS_DUAL && (io.evict_logits == nullptr || io.alive == nullptr)) code = BS_ERR_INVALID_ARG;
  else if ((T + g - 1) / g > MB || (T + s - 1) / s > rows || off < 0 ||
           (T + kPage - 1) / kPage > dims.max_pages_per_unit)
    code = BS_ERR_CAPACITY;
  else if (off % 4 != 0) code = BS_ERR_ALIGN;
  if (code != BS_OK) {
    drain();
    if (cj == 0) unit_error_publish(dims, io, words, u, code);
    return;
  }
  const Geom ge = unit_geom(T, g, s, sink, local);
  int n_tiles = 1;
  if (cls != BS_STREAMING) n_tiles = max(1, score_tiles(ge));
  const int n_ctas = (n_tiles + tpc - 1) / tpc;  // CTAs of this unit that take part
  float *score_row = io.scores + static_cast<size_t>(u) * MB;
  // Scored only when the candidates exist, in which case they start at the sink's end
  // and the rows copied above are this CTA's.
  const int my_tiles = (cls != BS_STREAMING && ge.c_hi > ge.c_lo) ? max(0, min(tpc, n_tiles - t0)) : 0;
  if (my_tiles > 0) {
    float *dots = reinterpret_cast<float *>(smem + L::off_dots(nbuf));
    ScoreQ<D, G> qf;
    for (int kk = 0; kk < my_tiles; ++kk) {
      const int bi = kk % nbuf;
      const int n_rows = inflight[bi];
      if (!wait_buf(bi)) {
        drain();
        return;
      }
      if (kk == 0) qf = score_qfrag<D, G>(qs);   // (the wait above was a CTA barrier)
      score_compute<D, G>(reinterpret_cast<const float *>(smem + bi * L::kTileBytes), qf, dots, ge, t0 + kk, reduce,
                          n_rows, score_row, [&] {
                            if (kk + nbuf < my_tiles)
                              inflight[bi] = score_copy<D>(summ, tile_row(t0 + kk + nbuf),
                                                           static_cast<int64_t>(ge.c_hi) * (g / s),
                                                           smem + bi * L::kTileBytes, &bars[bi]);
                          });
    }
  }
  if (!drain()) return;
  if (cj >= n_ctas) return;
  // ---- a1: the sub-block holding the appended token (first CTA, beside the others) --
  if (cj == 0 && tid < 32) unit_summary_update<D>(dims, kv, io, u, s, T, off, st);
  if (n_ctas > 1) {
    __syncthreads();
    if (tid == 0) is_last = (ticket_acq_rel(arrivals + u) == n_ctas - 1);
    __syncthreads();
    if (!is_last) return;
  }

  UnitFront uf;
  uf.u = u;
  uf.cls = cls;
  uf.k = k;
  uf.k_e = k_e;
  uf.g = g;
  uf.T = T;
  uf.ge = ge;
  unit_select_publish<kFrontThreads>(dims, kv, io, words, plist, pt_cache_ints, smem, sh, uf);
  if (tid == 0 && n_ctas > 1) arrivals[u] = 0;  // ready for the next step
}


// ---------------------------------------------------------------------------
// Fused step in the attention's workspace mode (more than 19 units with selections
// above 256 pages, or selections above 1024 pages) when a unit can have more than
// kFrontSelectMaxCandidates candidates: three launches, each a programmatic dependent
// of the one before. (With fewer, the front kernel above selects: two launches.)
//   1. step_score_balanced: a persistent grid; the score tiles (64 summary rows) of
//      every retrieval and dual unit, in unit order, form one stream cut into equal
//      contiguous shares, one per CTA; a CTA streams its tiles through a ring of nbuf
//      buffers (the next tiles' bulk copies fly during this tile's dot products, across
//      units).
//   2. step_select_kernel: one CTA per unit: a1 (one warp, while the others wait), a3,
//      the published count and a5. Streaming units need no scores and go ahead at
//      once; the others wait for launch 1 to finish.
//   3. the attention (workspace mode), which waits per unit for the published count.
// ---------------------------------------------------------------------------
constexpr int kMaxFrontRing = 3;   // tile buffers of the stream score kernel, at most

// A unit's head configuration, length and geometry for the step kernels.
struct FrontUnit {
  int cls, g, s, k, k_e, sink, local, T, rows;
  int64_t off;
  Geom ge;
  int code;    // BS_OK or the rule the unit breaks
  int tiles;   // score tiles (0: the unit is selected without scores)
};

__device__ __forceinline__ FrontUnit load_front_unit(const bs_dims &dims, const bs_kv &kv, const bs_head_cfg &cfg,
                                                     const bs_step_io &io, int u) {
  FrontUnit f;
  f.cls = cfg.cls[u];
  f.g = cfg.block_tokens[u];
  f.s = cfg.sub_tokens[u];
  f.k = cfg.k_total[u];
  f.k_e = cfg.k_evict[u];
  f.sink = cfg.sink_tokens[u];
  f.local = cfg.local_tokens[u];
  f.off = cfg.sum_off[u];
  f.rows = cfg.sum_rows[u];
  f.T = kv.seq_lens[u / dims.n_kv_heads];
  f.code = BS_OK;
  f.tiles = 0;
  if (!unit_cfg_ok(f.cls, f.g, f.s, f.k, f.k_e, f.sink, f.local) || f.T < 1) f.code = BS_ERR_INVALID_ARG;
  else if (f.cls == BS_DUAL && (io.evict_logits == nullptr || io.alive == nullptr)) f.code = BS_ERR_INVALID_ARG;
  else if ((f.T + f.g - 1) / f.g > dims.max_blocks_per_unit || (f.T + f.s - 1) / f.s > f.rows || f.off < 0 ||
           (f.T + kPage - 1) / kPage > dims.max_pages_per_unit)
    f.code = BS_ERR_CAPACITY;
  else if (f.off % 4 != 0) f.code = BS_ERR_ALIGN;
  if (f.code == BS_OK) {
    f.ge = unit_geom(f.T, f.g, f.s, f.sink, f.local);
    if (f.cls != BS_STREAMING && f.ge.c_hi > f.ge.c_lo) f.tiles = score_tiles(f.ge);
  }
  return f;
}

template <int D, int G>
__global__ void __launch_bounds__(kFrontThreads, 2) step_score_balanced(bs_dims dims, bs_kv kv, bs_head_cfg cfg,
                                                                     bs_step_io io, int reduce, int plan_off,
                                                                     int nbuf) {
  using L = ScoreLayout<D, G>;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t bars[kMaxFrontRing];
  __shared__ int scan_tmp[kFrontThreads / 32];
  const int tid = threadIdx.x, warp = tid >> 5;
  const int U = dims.batch * dims.n_kv_heads;
  const int P = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  int32_t *st = io.dev_status;
  int *pos = reinterpret_cast<int *>(smem + plan_off);   // [U + 1] first tile of unit u in the stream
  pdl_wait_front();    // q, lengths, KV pages and summaries are final
  pdl_trigger_front(); // the selection may start launching

  // ---- plan: tiles per unit, their offsets in the stream ------------------------------
  {
    const int per = (U + kFrontThreads - 1) / kFrontThreads;
    const int u0 = tid * per, u1 = min(U, u0 + per);
    int mine = 0;
    for (int u = u0; u < u1; ++u) {
      const int n = load_front_unit(dims, kv, cfg, io, u).tiles;
      pos[u] = n;   // a count for now (each thread owns its units' entries)
      mine += n;
    }
    int total;
    int run = front_scan(mine, scan_tmp, &total);
    for (int u = u0; u < u1; ++u) {
      const int n = pos[u];
      pos[u] = run;
      run += n;
    }
    if (tid == 0) {
      pos[U] = total;
      for (int i = 0; i < nbuf; ++i) mbar_init(&bars[i], 1);
      fence_mbar_init();
    }
    __syncthreads();
  }
  const int W = pos[U];
  const int Pe = min(P, W);
  const int p0 = c < Pe ? static_cast<int>(static_cast<int64_t>(W) * c / Pe) : 0;
  const int p1 = c < Pe ? static_cast<int>(static_cast<int64_t>(W) * (c + 1) / Pe) : 0;

  // ---- the share's tiles: tile t of unit u for t in [first_tile(u), end_tile(u)) ------
  float *qs = reinterpret_cast<float *>(smem + L::off_q(nbuf));
  float *dots = reinterpret_cast<float *>(smem + L::off_dots(nbuf));
  auto first_tile = [&](int u) { return max(p0, pos[u]) - pos[u]; };
  auto end_tile = [&](int u) { return min(p1, pos[u + 1]) - pos[u]; };
  int issue_u = p0 < p1 ? stream_rank_at(pos, U, p0) : U;
  int issue_t = issue_u < U ? first_tile(issue_u) : 0;
  int comp_u = issue_u, comp_t = issue_t;
  // The issuing unit's summary rows: its first candidate row and the end of its rows.
  const float *iss_summ = nullptr;
  int64_t iss_row0 = 0, iss_end = 0;
  int iss_for = -1;
  int inflight[kMaxFrontRing] = {0, 0, 0}, uses[kMaxFrontRing] = {0, 0, 0};
  auto issue_next = [&](int bi) {
    if (issue_u >= U || pos[issue_u] >= p1) {
      inflight[bi] = 0;
      return;
    }
    if (iss_for != issue_u) {
      const FrontUnit f = load_front_unit(dims, kv, cfg, io, issue_u);
      const int r = f.g / f.s;
      iss_summ = io.summaries + f.off;
      iss_row0 = static_cast<int64_t>(f.ge.c_lo) * r;
      iss_end = static_cast<int64_t>(f.ge.c_hi) * r;
      iss_for = issue_u;
    }
    if (tid == 0) fence_proxy_async_smem();   // the buffer's last reads come before the copy's writes
    inflight[bi] = score_copy<D>(iss_summ, iss_row0 + static_cast<int64_t>(issue_t) * kTileRows, iss_end,
                                 smem + bi * L::kTileBytes, &bars[bi]);
    if (++issue_t >= end_tile(issue_u)) {
      do {
        ++issue_u;
      } while (issue_u < U && pos[issue_u] < p1 && pos[issue_u + 1] == pos[issue_u]);   // units without tiles
      if (issue_u < U) issue_t = first_tile(issue_u);
    }
  };
  for (int i = 0; i < nbuf; ++i) issue_next(i);

  int q_u = -1;
  Geom cge;
  ScoreQ<D, G> qf;
  for (int n_done = 0; comp_u < U && pos[comp_u] < p1; ++n_done) {
    const int bi = n_done % nbuf;
    if (comp_u != q_u) {   // a new unit: its geometry and its queries (scaled) into shared memory
      q_u = comp_u;
      cge = load_front_unit(dims, kv, cfg, io, comp_u).ge;
      __syncthreads();     // the previous unit's tile is no longer read
      const int b = comp_u / dims.n_kv_heads, hk = comp_u % dims.n_kv_heads;
      const size_t qbase = (static_cast<size_t>(b) * dims.n_q_heads + static_cast<size_t>(hk) * G) * D;
      const void *qrow = dims.q_dtype == BS_BF16
                             ? static_cast<const void *>(static_cast<const uint16_t *>(io.q) + qbase)
                             : static_cast<const void *>(static_cast<const float *>(io.q) + qbase);
      score_load_q<D, G>(qs, qrow, dims.q_dtype);
      __syncthreads();
      qf = score_qfrag<D, G>(qs);
    }
    const int n_rows = inflight[bi];
    const bool ok = score_wait(&bars[bi], static_cast<uint32_t>(uses[bi] & 1), n_rows, st);
    if (n_rows > 0) ++uses[bi];
    inflight[bi] = 0;
    if (!ok) break;   // (reported) a copy that never landed: no more tiles
    score_compute<D, G>(reinterpret_cast<const float *>(smem + bi * L::kTileBytes), qf, dots, cge, comp_t, reduce,
                        n_rows, io.scores + static_cast<size_t>(comp_u) * dims.max_blocks_per_unit,
                        [&] { issue_next(bi); });
    if (++comp_t >= end_tile(comp_u)) {
      do {
        ++comp_u;
      } while (comp_u < U && pos[comp_u] < p1 && pos[comp_u + 1] == pos[comp_u]);
      if (comp_u < U) comp_t = first_tile(comp_u);
    }
  }
  // Whatever is still in flight lands before the CTA exits.
  for (int i = 0; i < nbuf; ++i)
    if (inflight[i] > 0) score_wait(&bars[i], static_cast<uint32_t>(uses[i] & 1), inflight[i], st);
}

// One CTA per unit: the selection (a3), its page list, the published count and the
// set-difference (a5). A streaming unit needs no scores and goes ahead at once; the
// others wait for the score kernel (and everything before it) to finish.
constexpr int kStepSelThreads = 1024;   // at most 8 candidates per thread in registers up to 8192

template <int D>
__global__ void __launch_bounds__(kStepSelThreads) step_select_kernel(bs_dims dims, bs_kv kv, bs_head_cfg cfg,
                                                                    bs_step_io io, StepWords words, int32_t *plist,
                                                                    int pt_cache_ints) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ SelShared<kStepSelThreads> sh;
  const int u = blockIdx.x;
  pdl_trigger_front();   // the attention may start launching
  const FrontUnit f = load_front_unit(dims, kv, cfg, io, u);
  // a1 by warp 0 while the others wait for the scores: the sub-block holding the
  // appended token lies in the always-forced tail block, which no score of this step
  // reads, and its K pages were written before the score kernel started.
  if (f.code == BS_OK && threadIdx.x < 32) unit_summary_update<D>(dims, kv, io, u, f.s, f.T, f.off, io.dev_status);
  if (f.code != BS_OK || f.cls != BS_STREAMING) pdl_wait_front();
  if (f.code != BS_OK) {
    unit_error_publish(dims, io, words, u, f.code);
    return;
  }
  UnitFront uf;
  uf.u = u;
  uf.cls = f.cls;
  uf.k = f.k;
  uf.k_e = f.k_e;
  uf.g = f.g;
  uf.T = f.T;
  uf.ge = f.ge;
  unit_select_publish<kStepSelThreads>(dims, kv, io, words, plist, pt_cache_ints, smem, sh, uf);
}

bs_status launch_step_attention(const bs_dims &dims, const bs_kv &kv, const bs_head_cfg &cfg, const bs_step_io &io,
                                cudaStream_t cs, const StepWords &words, int32_t *plist, int mode);

template <int D, int G>
bs_status launch_step(const bs_dims &dims, const bs_kv &kv, const bs_head_cfg &cfg, const bs_step_io &io,
                      int reduce, cudaStream_t cs) {
  constexpr size_t kFrontMaxSmem = 200 * 1024;
  static const bool attr_ok = cudaFuncSetAttribute(step_front_kernel<D, G>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(kFrontMaxSmem)) == cudaSuccess;
  if (!attr_ok) return BS_ERR_CUDA;
  const int units = dims.batch * dims.n_kv_heads;
  const int mode = attn_mode(units, dims.max_gather_pages_per_unit);
  const bool lists = mode != kModeWorkspace;   // the attention reads page lists
  int pt_cache = lists && dims.max_pages_per_unit <= kPtCacheInts ? dims.max_pages_per_unit : 0;
  size_t front_smem = front_select_bytes(dims.max_blocks_per_unit, dims.max_sel_per_unit, pt_cache);
  if (front_smem > kFrontMaxSmem) {  // read the page table from global memory instead
    pt_cache = 0;
    front_smem = front_select_bytes(dims.max_blocks_per_unit, dims.max_sel_per_unit, 0);
  }
  const StepWords words = step_words(io.workspace, units);
  int32_t *plist = lists ? words.tickets + attn_counter_floats(units) : nullptr;
  if (step_selects_apart(units, dims.max_gather_pages_per_unit, dims.max_blocks_per_unit)) {
    // 1. scores in equal shares: the ring of nbuf score tiles, the queries and dot products,
    //    then the plan; nbuf 2 or 3, whichever gives more tiles in flight per SM
    //    (preferring more CTAs).
    static const bool sc_ok = cudaFuncSetAttribute(step_score_balanced<D, G>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(kFrontMaxSmem)) == cudaSuccess &&
                              cudaFuncSetAttribute(step_select_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(kFrontMaxSmem)) == cudaSuccess;
    if (!sc_ok) return BS_ERR_CUDA;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return BS_ERR_CUDA;
    int best_nbuf = 0, best_per_sm = 0, best_plan = 0;
    size_t best_smem = 0;
    for (int nb = kMaxFrontRing; nb >= 2; --nb) {
      const size_t plan_off = (static_cast<size_t>(ScoreLayout<D, G>::bytes(nb)) + 15) & ~size_t(15);
      const size_t smem = plan_off + (static_cast<size_t>(units) + 1) * 4;
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, step_score_balanced<D, G>, kFrontThreads, smem) !=
              cudaSuccess ||
          per_sm <= 0)
        continue;
      if (per_sm * nb > best_per_sm * best_nbuf || (per_sm * nb == best_per_sm * best_nbuf && per_sm > best_per_sm)) {
        best_nbuf = nb;
        best_per_sm = per_sm;
        best_plan = static_cast<int>(plan_off);
        best_smem = smem;
      }
    }
    if (best_nbuf == 0) return BS_ERR_CAPACITY;
    if (launch_ex(step_score_balanced<D, G>, dim3(best_per_sm * sms), kFrontThreads, best_smem, cs, 0, true, dims,
                  kv, cfg, io, reduce, best_plan, best_nbuf) != cudaSuccess)
      return BS_ERR_CUDA;
    // 2. selection, one CTA per unit.
    if (launch_ex(step_select_kernel<D>, dim3(units), kStepSelThreads, front_smem, cs, 0, true, dims, kv, cfg, io, words,
                  plist, pt_cache) != cudaSuccess)
      return BS_ERR_CUDA;
    // 3. attention.
    return launch_step_attention(dims, kv, cfg, io, cs, words, plist, mode);
  }
  // Score tiles per CTA: one while the launch fits about two waves of two CTAs per SM
  // (short, latency-bound steps); more for large steps, up to 8, so that each CTA
  // streams several tiles through two buffers and the grid stays near one wave.
  const int max_tiles = dims.max_subs_per_unit / kTileRows + 2;
  const long long work = static_cast<long long>(units) * max_tiles;
  const int slots = attn_target_ctas();
  const int tpc = static_cast<int>(std::min<long long>(8, std::max<long long>(1, (work + 2 * slots - 1) / (2 * slots))));
  const int nbuf = tpc > 1 ? 2 : 1;
  if (front_smem < static_cast<size_t>(ScoreLayout<D, G>::bytes(nbuf))) front_smem = ScoreLayout<D, G>::bytes(nbuf);
  if (front_smem > kFrontMaxSmem) return BS_ERR_CAPACITY;
  const dim3 front_grid(units, (max_tiles + tpc - 1) / tpc);
  if (launch_ex(step_front_kernel<D, G>, front_grid, kFrontThreads, front_smem, cs, 0, true, dims, kv, cfg, io,
                reduce, words, plist, pt_cache, tpc) != cudaSuccess)
    return BS_ERR_CUDA;
  return launch_step_attention(dims, kv, cfg, io, cs, words, plist, mode);
}

// The attention of the fused step, a programmatic dependent of the front kernel.
bs_status launch_step_attention(const bs_dims &dims, const bs_kv &kv, const bs_head_cfg &cfg, const bs_step_io &io,
                                cudaStream_t cs, const StepWords &words, int32_t *plist, int mode) {
  const int units = dims.batch * dims.n_kv_heads;
  AttnArgs a;
  a.dims = dims;
  a.q = io.q;
  a.kv = kv;
  a.cfg = cfg;
  a.sel_idx = io.cur_idx;
  a.sel_cnt = io.cur_cnt;
  a.bias = io.evict_bias;
  a.out = io.out;
  a.lse = io.lse;
  a.arrivals = words.arrivals;
  a.records = static_cast<float *>(io.workspace) + attn_records_offset(units);
  a.plist = plist;
  a.pub = words.pub;
  a.expect = words.expect;
  a.st = io.dev_status;
  a.wait_ns = wait_limit_ns();
  return dims.kv_dtype == BS_BF16 ? launch_attn_bf16(a, true, cs) : launch_attn_f32(a, true, cs);
}

template <int D>
bs_status dispatch_g(int G, const bs_dims &dims, const bs_kv &kv, const bs_head_cfg &cfg, const bs_step_io &io,
                     int reduce, cudaStream_t cs) {
  switch (G) {
    case 1: return launch_step<D, 1>(dims, kv, cfg, io, reduce, cs);
    case 2: return launch_step<D, 2>(dims, kv, cfg, io, reduce, cs);
    case 3: return launch_step<D, 3>(dims, kv, cfg, io, reduce, cs);
    case 4: return launch_step<D, 4>(dims, kv, cfg, io, reduce, cs);
    case 5: return launch_step<D, 5>(dims, kv, cfg, io, reduce, cs);
    case 6: return launch_step<D, 6>(dims, kv, cfg, io, reduce, cs);
    case 7: return launch_step<D, 7>(dims, kv, cfg, io, reduce, cs);
    default: return launch_step<D, 8>(dims, kv, cfg, io, reduce, cs);
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
  if (dims->head_dim == 128) return dispatch_g<128>(G, *dims, *kv, *cfg, *io, group_reduce, cs);
  return dispatch_g<64>(G, *dims, *kv, *cfg, *io, group_reduce, cs);
}
