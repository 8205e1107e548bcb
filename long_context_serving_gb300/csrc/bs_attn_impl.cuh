// Device code of the sparse decode attention (a4), shared by the stand-alone kernel and
// the fused decode step ("Technische Samenvatting: Fluxion", Probleemstelling item 1:
// top-k selection, then sparse attention over the selected KV blocks; Kerninzichten
// item 3: this work is bound by data movement).
//
// Split-KV flash-decode. A unit's selected blocks cover n_pages pages of 16 tokens,
// cut into splits of pps pages: in cluster mode (selections up to 1024 pages) S splits
// per unit, S the largest power of two up to 16 that keeps the launch in one wave of
// about two CTAs per SM, pps = ceil(n_pages / S); in workspace mode up to 32 splits of
// a multiple of 4 pages. One CTA per (split, unit):
//   * the unit's page-table row is pulled into L2 while the selection count and row are
//     read into shared memory; warp 0 resolves the split's pages 32 at a time and stages
//     them into a ring of 4-page stages (for bf16 three deep in cluster mode and two
//     in workspace mode, with three CTAs per SM; two for fp32) with TMA
//     copies that complete an mbarrier with their byte count;
//   * bf16 caches (attn_split_mma, 4 warps): each warp takes one 16-token page per
//     stage. Pages arrive through a tiled tensor map with 128-byte swizzle, so
//     ldmatrix reads them without bank conflicts. q.K and P.V are warp-level bf16
//     tensor-core MMAs (m16n8k16, fp32 accumulate) with the query heads as the rows:
//     q and K are exact in bf16; P stays in registers and enters P.V as a bf16 pair
//     hi + lo (hi = bf16(p), lo = bf16(p - hi)), which keeps it to about 2^-16
//     relative. Online softmax per head in fp32 with base-2 exponents; the four
//     warps' states are combined at the end;
//   * fp32 caches (attn_split_ffma, 8 warps): 1-D bulk copies; q.K with four threads
//     per token over rotated 16-byte chunks, one warp per head for the softmax, and
//     P.V with lanes owning head_dim/32 dimensions;
//   * merge, cluster mode: a unit's S splits are one thread-block cluster; each keeps
//     its (o, m, l) in shared memory and, after a cluster barrier, each CTA merges a
//     slice of the output by log-sum-exp reading its peers' shared memory (no global
//     traffic, no atomics); a single split normalises its own state;
//   * merge, workspace mode: a unit with one split writes its output directly;
//     otherwise each split writes an (o, m, l) record and takes an arrival ticket (one
//     acquire-release atomic per CTA); the last split merges the records in split order.
// Tokens past T inside a partial tail page are masked out of both products.
//
// In step mode (the fused decode step, launched as a programmatic dependent of the
// selection kernel) a streaming unit's blocks are its forced blocks, computed from the
// geometry, so its splits run without waiting; every other unit waits (bounded) until
// the selection kernel has published that unit's selection count with a release
// store, then reads its pages from the page list the selection kernel wrote (cluster
// mode) or its row.
#pragma once

#include <cuda.h>
#include <math.h>

#include "bs_attn_launch.cuh"
#include "bs_attn_plan.cuh"
#include "bs_internal.cuh"

namespace bsi {

constexpr float kLog2e = 1.4426950408889634f;

// A CTA's unit and split. The grid is (splits, units) in cluster mode, where a unit's
// splits form one cluster along x, and (units, splits) in workspace mode, so that every
// unit's first split is dispatched before any unit's second: in the fused step a unit
// whose selection is published early does not queue behind the splits of units still
// being selected.
__device__ __forceinline__ int attn_unit_id(bool in_cluster) {
  return static_cast<int>(in_cluster ? blockIdx.y : blockIdx.x);
}
__device__ __forceinline__ int attn_split_id(bool in_cluster) {
  return static_cast<int>(in_cluster ? blockIdx.x : blockIdx.y);
}
__device__ __forceinline__ int attn_n_splits(bool in_cluster) {
  return static_cast<int>(in_cluster ? gridDim.x : gridDim.y);
}
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kSelPreload = 512;  // selection entries staged in shared memory
constexpr int kMmaThreads = 128;  // bf16 path: 4 warps, one page each per stage

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ int load_relaxed_gpu(const int32_t *p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Starts pulling unit u's page-table row into L2 (one 128-byte line per thread) while
// the block list is read, so the page lookups that follow hit L2. Skipped when the
// fused step hands the attention its pages ready in a page list.
template <int NT>
__device__ __forceinline__ void prefetch_page_row(const bs_dims &dims, const bs_kv &kv, const bs_head_cfg &cfg,
                                                  const int32_t *plist, int u, bool in_step) {
  if (plist != nullptr && in_step && cfg.cls[u] != BS_STREAMING) return;
  const int32_t *row = kv.page_table + static_cast<size_t>(u) * dims.max_pages_per_unit;
  const int lines = (dims.max_pages_per_unit + 31) / 32;
  for (int i = threadIdx.x; i < lines; i += NT) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + i * 32));
}

__device__ __forceinline__ int atomic_add_acq_rel_gpu(int32_t *p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// ---------------------------------------------------------------------------
// The block list of one unit as the attention sees it.
// ---------------------------------------------------------------------------
struct UnitBlocks {
  bool ok;
  int T, g, cnt;
  bool computed;          // forced blocks from the geometry (streaming unit, step mode)
  int n_sink, lo2;        // computed list: [0, n_sink) then [lo2, lo2 + cnt - n_sink)
  const int32_t *sel;     // selection row (global), when not computed
  const int32_t *sel_sm;  // its first kSelPreload entries in shared memory
  const int32_t *plist;   // the unit's page list (fused step), or null
  bool polled;            // the count came from the fused step's published word
  int epoch;              // the epoch that word carried
  UnitPages pg;

  __device__ __forceinline__ int block(int i) const {
    if (computed) return i < n_sink ? i : lo2 + (i - n_sink);
    return i < kSelPreload ? sel_sm[i] : sel[i];
  }
};

// Reads a unit's block list (waiting for the selection kernel in step mode unless
// the unit is streaming) and its split plan. All NT threads call it.
// Waits (bounded by wait_ns) until the fused step's front kernel has published unit
// u's selection for this step: the published word carries the epoch after the one in
// expect[u] (which the attention advances once every reader of the unit is done).
// Returns the count, or 0 after reporting BS_ERR_TIMEOUT; *epoch gets the epoch.
// Relaxed polls with a short sleep, then one acquire fence, so the row and the page
// list written before the release store are visible.
__device__ __forceinline__ int wait_published(const int32_t *pub, const int32_t *expect, int u, uint64_t wait_ns,
                                              int32_t *st, int *epoch) {
  const int e = (__ldcg(expect + u) + 1) & kEpochMask;
  *epoch = e;
  int w = load_relaxed_gpu(pub + u);
  if ((w >> 16) != e) {
    const uint64_t t0 = global_ns();
    while (((w = load_relaxed_gpu(pub + u)) >> 16) != e) {
      __nanosleep(64);
      if (global_ns() - t0 > wait_ns) {
        report(st, BS_ERR_TIMEOUT);
        return 0;
      }
    }
  }
  fence_acq_rel_gpu();
  return w & 0xffff;
}

template <int NT>
__device__ UnitBlocks load_unit_blocks(const AttnArgs &a, int u, int32_t *sel_sm, bool in_step, bool in_cluster) {
  const bs_dims &dims = a.dims;
  const bs_kv &kv = a.kv;
  const bs_head_cfg &cfg = a.cfg;
  const int32_t *sel_idx = a.sel_idx, *sel_cnt = a.sel_cnt, *plist = a.plist;
  int32_t *st = a.st;
  __shared__ int sh_cnt;
  const int tid = threadIdx.x, split = attn_split_id(in_cluster);
  const int b = u / dims.n_kv_heads;
  UnitBlocks ub;
  ub.T = kv.seq_lens[b];
  ub.g = cfg.block_tokens[u];
  ub.computed = false;
  ub.sel = sel_idx + static_cast<size_t>(u) * dims.max_sel_per_unit;
  ub.sel_sm = sel_sm;
  ub.plist = nullptr;
  ub.polled = false;
  ub.epoch = 0;
  ub.n_sink = ub.lo2 = 0;
  ub.cnt = 0;
  const bool cfg_ok = ub.g > 0 && ub.g % kPage == 0 && ub.T >= 1;
  if (in_step && cfg.cls[u] == BS_STREAMING && cfg_ok) {
    const Geom ge = unit_geom(ub.T, ub.g, cfg.sub_tokens[u], cfg.sink_tokens[u], cfg.local_tokens[u]);
    ub.computed = true;
    ub.n_sink = ge.n_sink;
    ub.lo2 = ge.local_lo > ge.n_sink ? ge.local_lo : ge.n_sink;
    ub.cnt = ge.n_sink + (ge.n_blk - ub.lo2);
  }
  if (!ub.computed && !in_step) {
    // The count and the first entries of the row are read together (entries past the
    // count are never used).
    const int ns = min(dims.max_sel_per_unit, kSelPreload);
    if (tid == 0) sh_cnt = sel_cnt[u];
    for (int i = tid; i < ns; i += NT) sel_sm[i] = ub.sel[i];
    __syncthreads();
    ub.cnt = sh_cnt;
  } else if (!ub.computed) {
    __shared__ int sh_epoch;
    if (tid == 0) {
      int e = 0;
      sh_cnt = wait_published(a.pub, a.expect, u, a.wait_ns, st, &e);
      sh_epoch = e;
    }
    __syncthreads();
    ub.cnt = sh_cnt;
    ub.polled = true;
    ub.epoch = sh_epoch;
    if (plist != nullptr) {
      // The selection kernel also wrote the pages of the selected blocks; the last
      // selected block is the tail block, which is always forced.
      ub.plist = plist + static_cast<size_t>(u) * dims.max_gather_pages_per_unit;
    } else {
      const int ns = min(min(dims.max_sel_per_unit, kSelPreload), max(ub.cnt, 0));
      for (int i = tid; i < ns; i += NT) sel_sm[i] = __ldcg(ub.sel + i);
      __syncthreads();
    }
  }
  ub.ok = cfg_ok && ub.cnt >= 0 && ub.cnt <= dims.max_sel_per_unit;
  if (!ub.ok && split == 0 && tid == 0) report(st, BS_ERR_INVALID_ARG);
  int last = -1;
  if (ub.ok && ub.cnt > 0) {
    last = ub.plist ? (ub.T - 1) / ub.g : ub.block(ub.cnt - 1);
    if (last < 0 || static_cast<int64_t>(last) * ub.g >= ub.T) {
      if (split == 0 && tid == 0) report(st, BS_ERR_DEVICE_BOUNDS);
      ub.ok = false;
    }
  }
  ub.pg = unit_pages(ub.T, ub.g, ub.ok ? ub.cnt : 0, last, in_cluster ? static_cast<int>(gridDim.x) : 0,
                     attn_min_split_pages(dims.max_gather_pages_per_unit));
  if (ub.plist && ub.pg.n_pages > dims.max_gather_pages_per_unit) {
    if (split == 0 && tid == 0) report(st, BS_ERR_CAPACITY);
    ub.pg.n_pages = 0;
  }
  return ub;
}

// Splits of unit u that take part in the fused step's workspace-mode attention, from the
// head configuration and the length alone (every split of the unit computes the same
// number before any wait): a selection holds the forced blocks (sink, local window,
// tail) and at most k others, so its pages are at most min(n_blk, |F| + k) * g/16; with
// selections up to 1024 pages every split but the last holds at least kMidSplitPages
// pages, so ceil(pages / kMidSplitPages) bounds the split count. The splits past it can
// hold no page: they leave at once instead of holding an SM slot until the unit's
// selection is published. Any other case: every launched split.
__device__ __forceinline__ int step_ws_splits(const AttnArgs &a, int u, int launched) {
  const bs_dims &dims = a.dims;
  if (attn_min_split_pages(dims.max_gather_pages_per_unit) != kMidSplitPages) return launched;
  const bs_head_cfg &cfg = a.cfg;
  const int cls = cfg.cls[u], g = cfg.block_tokens[u], s = cfg.sub_tokens[u], k = cfg.k_total[u];
  const int sink = cfg.sink_tokens[u], local = cfg.local_tokens[u];
  if (!unit_cfg_ok(cls, g, s, k, cfg.k_evict[u], sink, local)) return launched;
  const int T = a.kv.seq_lens[u / dims.n_kv_heads];
  if (T < 1) return launched;
  const Geom ge = unit_geom(T, g, s, sink, local);
  const int n_forced = ge.n_sink + (ge.n_blk - max(ge.local_lo, ge.n_sink));
  const long long blocks =
      cls == BS_STREAMING ? n_forced : min(static_cast<long long>(ge.n_blk), static_cast<long long>(n_forced) + k);
  const long long pages = min(blocks * (g / kPage), static_cast<long long>(dims.max_gather_pages_per_unit));
  const int n = static_cast<int>((pages + kMidSplitPages - 1) / kMidSplitPages);
  return max(1, min(launched, n));
}

// A selection with more splits than take part would lose pages: it is reported
// (BS_ERR_DEVICE_BOUNDS) and the unit attends nothing rather than part of it.
__device__ __forceinline__ void check_split_bound(UnitBlocks &ub, int n_part, int split, int32_t *st) {
  if (ub.pg.n_split > n_part) {
    if (split == 0 && threadIdx.x == 0) report(st, BS_ERR_DEVICE_BOUNDS);
    ub.ok = false;
  }
}

// Resolves page slot `lane` (< kStagePages) of a stage: returns the physical page and
// the number of valid tokens in it (0 for an empty or out-of-range slot). blk_out (may
// be null) receives the page's block index, -1 for an empty slot.
__device__ __forceinline__ int resolve_page(const UnitBlocks &ub, const bs_dims &dims, const int32_t *pt, int gp,
                                            int gp1, int *phys_out, int *blk_out, int32_t *st) {
  *phys_out = -1;
  if (blk_out) *blk_out = -1;
  if (gp >= gp1) return 0;
  if (ub.plist) {
    // Pages come resolved; all are full but the unit's last, which holds token T-1.
    const int phys = __ldcg(ub.plist + gp);
    if (phys < 0 || phys >= dims.n_pages) {
      report(st, BS_ERR_DEVICE_BOUNDS);
      return 0;
    }
    *phys_out = phys;
    if (blk_out) *blk_out = __ldcg(ub.sel + gp / (ub.g / kPage));
    return gp == ub.pg.n_pages - 1 ? (ub.T - 1) % kPage + 1 : kPage;
  }
  const int ppb = ub.pg.ppb;
  const int i = gp / ppb, pb = gp - i * ppb;
  const int c = ub.block(i);
  if (blk_out) *blk_out = c;
  const int lp = c * ppb + pb;
  const int t0 = lp * kPage;
  if (c < 0 || lp >= dims.max_pages_per_unit || t0 >= ub.T) {
    report(st, BS_ERR_DEVICE_BOUNDS);
    return 0;
  }
  const int phys = __ldg(pt + lp);
  if (phys < 0 || phys >= dims.n_pages) {
    report(st, BS_ERR_DEVICE_BOUNDS);
    return 0;
  }
  *phys_out = phys;
  return min(kPage, ub.T - t0);
}

// The logit bias of block c of unit u in log2 units: 0 without biases (or for an empty
// slot), else log2(e) * bias[u][c] (a block index outside the row reports
// BS_ERR_DEVICE_BOUNDS and drops the page).
__device__ __forceinline__ float block_bias2(const float *bias, const bs_dims &dims, int u, int c, int32_t *st) {
  if (bias == nullptr || c < 0) return 0.0f;
  if (c >= dims.max_blocks_per_unit) {
    report(st, BS_ERR_DEVICE_BOUNDS);
    return -INFINITY;
  }
  return __ldg(bias + static_cast<size_t>(u) * dims.max_blocks_per_unit + c) * kLog2e;
}

// Output row of one head from an unnormalised state (o, m in log2 units, l): o / l and
// lse = ln 2 (m + log2 l); a state with l = 0 (nothing attended) gives a zero row and
// lse = -inf.
__device__ __forceinline__ void write_normalised(float4 o, float m, float l, float *orow, float *lse_h, int dq) {
  if (l > 0.0f) {
    const float inv = 1.0f / l;
    o.x *= inv; o.y *= inv; o.z *= inv; o.w *= inv;
  } else {
    o = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  reinterpret_cast<float4 *>(orow)[dq] = o;
  if (dq == 0) *lse_h = l > 0.0f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

// Epilogue of the workspace mode, shared by both paths. `o_sm` holds this split's
// unnormalised output [G][D] (fp32, shared), `m_sm`/`l_sm` its per-head max (log2
// units) and sum. With one taking part (`ns`, the splits of the unit that take part:
// every launched one, or step_ws_splits in the fused step) it writes out/lse; otherwise
// every split taking part (an idle one with an empty state) publishes its record and
// takes a ticket, and the last of them merges the records in split order and, in the
// fused step, advances the unit's epoch (every split taking part has read it by then).
// `scratch` needs 3 * kMaxG * kAttnMaxSplits floats of shared memory. All NT threads
// call it.
template <int NT, int D, int G>
__device__ void finish_split(const UnitBlocks &ub, int u, size_t orow0, const float *o_sm, const float *m_sm,
                             const float *l_sm, int32_t *arrivals, float *ws, float *out, float *lse, float *scratch,
                             int32_t *expect, int ns) {
  constexpr int QD = D / 4;
  constexpr int REC = attn_record_floats(D);
  __shared__ int is_last;
  __shared__ float ML[2][kMaxG];
  // (workspace mode: the grid is (units, splits), attn_split_id)
  const int tid = threadIdx.x, split = attn_split_id(false);
  if (ns == 1) {
    for (int i = tid; i < G * QD; i += NT) {
      const int h = i / QD, dq = i % QD;
      write_normalised(reinterpret_cast<const float4 *>(o_sm + h * D)[dq], m_sm[h], l_sm[h], out + (orow0 + h) * D,
                       lse + orow0 + h, dq);
    }
    if (ub.polled && tid == 0) expect[u] = ub.epoch;
    return;
  }
  float *rec = ws + (static_cast<size_t>(u) * kAttnMaxSplits + split) * G * REC;
  for (int i = tid; i < G * QD; i += NT) {
    const int h = i / QD, dq = i % QD;
    reinterpret_cast<float4 *>(rec + h * REC)[dq] = reinterpret_cast<const float4 *>(o_sm + h * D)[dq];
  }
  if (tid < G) {
    rec[tid * REC + D] = m_sm[tid];
    rec[tid * REC + D + 1] = l_sm[tid];
  }
  // Publish the record and take an arrival ticket: the CTA barrier orders every
  // thread's record writes before thread 0's release; the last split acquires.
  __syncthreads();
  if (tid == 0) is_last = (atomic_add_acq_rel_gpu(arrivals + u, 1) == ns - 1);
  __syncthreads();
  if (!is_last) return;
  // Merge: M = max m_i, L = sum l_i 2^(m_i - M), o = sum 2^(m_i - M) o_i / L,
  // lse = ln 2 (M + log2 L); splits are visited in index order.
  const float *base = ws + static_cast<size_t>(u) * kAttnMaxSplits * G * REC;
  float *m_all = scratch;                          // [G][32]
  float *l_all = m_all + kMaxG * kAttnMaxSplits;
  float *w_all = l_all + kMaxG * kAttnMaxSplits;
  for (int i = tid; i < G * ns; i += NT) {
    const int h = i / ns, sp = i % ns;
    const float *r = base + (static_cast<size_t>(sp) * G + h) * REC;
    m_all[h * kAttnMaxSplits + sp] = __ldcg(r + D);
    l_all[h * kAttnMaxSplits + sp] = __ldcg(r + D + 1);
  }
  __syncthreads();
  if (tid < G) {
    float M = -INFINITY;
    for (int sp = 0; sp < ns; ++sp) M = fmaxf(M, m_all[tid * kAttnMaxSplits + sp]);
    float Lsum = 0.0f;
    for (int sp = 0; sp < ns; ++sp) {
      const float mi = m_all[tid * kAttnMaxSplits + sp];
      const float w = (mi == -INFINITY) ? 0.0f : exp2f(mi - M);
      w_all[tid * kAttnMaxSplits + sp] = w;
      Lsum = fmaf(l_all[tid * kAttnMaxSplits + sp], w, Lsum);
    }
    ML[0][tid] = M;
    ML[1][tid] = Lsum;
  }
  __syncthreads();
  constexpr int kBatch = 8;
  for (int i = tid; i < G * QD; i += NT) {
    const int h = i / QD, dq = i % QD;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp0 = 0; sp0 < ns; sp0 += kBatch) {
      float4 v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (sp0 + j < ns)
          v[j] = __ldcg(reinterpret_cast<const float4 *>(base + (static_cast<size_t>(sp0 + j) * G + h) * REC) + dq);
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (sp0 + j < ns) {
          const float w = w_all[h * kAttnMaxSplits + sp0 + j];
          o.x = fmaf(v[j].x, w, o.x);
          o.y = fmaf(v[j].y, w, o.y);
          o.z = fmaf(v[j].z, w, o.z);
          o.w = fmaf(v[j].w, w, o.w);
        }
    }
    write_normalised(o, ML[0][h], ML[1][h], out + (orow0 + h) * D, lse + orow0 + h, dq);
  }
  if (tid == 0) {
    arrivals[u] = 0;  // ready for the next call
    if (ub.polled) expect[u] = ub.epoch;
  }
}

// ---------------------------------------------------------------------------
// Cluster-mode merge through distributed shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t peer_addr(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_peer(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_peer4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a)
               : "memory");
  return v;
}

// Every CTA of the cluster (C splits of one unit) holds its split's unnormalised
// o [G][D], m [G] (log2 units) and l [G] in shared memory (an idle split: m = -inf,
// l = 0, o = 0). After a cluster barrier CTA r merges float4 columns r, r + C, ... of
// the output over the C splits in split order (all peer loads of a column issued
// before their use); a second barrier keeps every CTA alive until its peers have read
// it. All threads of all CTAs of the cluster call it.
template <int NT, int D, int G, int C>
__device__ void cluster_merge_c(size_t orow0, const float *o_sm, const float *m_sm, const float *l_sm, float *out,
                                float *lse) {
  constexpr int QD = D / 4, NF4 = G * QD;
  cluster_sync_all();
  const uint32_t rank = cluster_rank();
  for (int i = static_cast<int>(rank) + C * static_cast<int>(threadIdx.x); i < NF4; i += C * NT) {
    const int h = i / QD, dq = i % QD;
    float mp[C], lp[C];
    float M = -INFINITY;
#pragma unroll
    for (int p = 0; p < C; ++p) {
      mp[p] = ld_peer(peer_addr(m_sm + h, p));
      lp[p] = ld_peer(peer_addr(l_sm + h, p));
      M = fmaxf(M, mp[p]);
    }
    float4 v[C];
#pragma unroll
    for (int p = 0; p < C; ++p) v[p] = ld_peer4(peer_addr(o_sm + h * D + dq * 4, p));
    float Lsum = 0.0f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int p = 0; p < C; ++p) {
      const float w = (mp[p] == -INFINITY) ? 0.0f : exp2f(mp[p] - M);
      Lsum = fmaf(lp[p], w, Lsum);
      o.x = fmaf(v[p].x, w, o.x);
      o.y = fmaf(v[p].y, w, o.y);
      o.z = fmaf(v[p].z, w, o.z);
      o.w = fmaf(v[p].w, w, o.w);
    }
    write_normalised(o, M, Lsum, out + (orow0 + h) * D, lse + orow0 + h, dq);
  }
  cluster_sync_all();
}

// Merge of the C = gridDim.x splits of a cluster (a power of two up to 16); a single
// split normalises its own state.
template <int NT, int D, int G>
__device__ void cluster_merge(size_t orow0, const float *o_sm, const float *m_sm, const float *l_sm, float *out,
                              float *lse) {
  constexpr int QD = D / 4, NF4 = G * QD;
  switch (gridDim.x) {
    case 2: cluster_merge_c<NT, D, G, 2>(orow0, o_sm, m_sm, l_sm, out, lse); return;
    case 4: cluster_merge_c<NT, D, G, 4>(orow0, o_sm, m_sm, l_sm, out, lse); return;
    case 8: cluster_merge_c<NT, D, G, 8>(orow0, o_sm, m_sm, l_sm, out, lse); return;
    case 16: cluster_merge_c<NT, D, G, 16>(orow0, o_sm, m_sm, l_sm, out, lse); return;
    default: break;
  }
  for (int i = threadIdx.x; i < NF4; i += NT) {
    const int h = i / QD, dq = i % QD;
    write_normalised(reinterpret_cast<const float4 *>(o_sm + h * D)[dq], m_sm[h], l_sm[h], out + (orow0 + h) * D,
                     lse + orow0 + h, dq);
  }
}

// ===========================================================================
// bf16 path: tiled TMA + warp-level tensor-core MMA
// ===========================================================================
template <int D>
struct MmaLayout {
  static constexpr int kRingMax = 3;                   // stages in flight, at most
  static constexpr int kHalves = D / 64;               // 128-byte-wide column halves of a row
  static constexpr int kHalfBytes = kPage * 128;       // 16 rows x 128 B = 2 KiB (swizzle atom x2)
  static constexpr int kPageBytes = kHalves * kHalfBytes;
  static constexpr int kStageKV = kStagePages * kPageBytes;  // K (or V) of one stage
  static constexpr int kBufBytes = 2 * kStageKV;              // K then V
  // `ring` stage buffers, then the staged selection entries.
  __host__ __device__ static constexpr int off_sel(int ring) { return ring * kBufBytes; }
  __host__ __device__ static constexpr int bytes(int ring) { return off_sel(ring) + kSelPreload * 4; }
  // After the last stage: warp states [4][8][D] and (m, l) reuse buffer 0; the merge's
  // scratch reuses buffer 1.
  static_assert(4 * kMaxG * D * 4 + 2 * 4 * kMaxG * 4 <= kBufBytes, "combine scratch");
  static_assert(3 * kMaxG * kAttnMaxSplits * 4 <= kBufBytes, "merge scratch");
};

// Stages in flight per CTA: three in cluster mode; two in workspace mode, where a third
// CTA per SM (more splits resident while units wait for their selections) pays more.
__host__ __device__ constexpr int attn_mma_ring(bool cluster) { return cluster ? 3 : 2; }

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D = A B + D for m16n8k16, bf16 inputs, fp32 accumulators (row-major A, column-major B).
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Transpose of an 8x8 matrix of 16-bit values held one register per thread in the MMA
// fragment layout (row lane/4, columns 2(lane%4), 2(lane%4)+1).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float bf16_lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Byte offset of 16-byte chunk `c` (0..D/8-1) of row `r` (0..15) inside a page tile
// written by a 128-byte-swizzled TMA box per column half.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * (kPage * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// The G query rows of a unit (starting at row orow0 of q) as MMA A fragments of one
// warp: rows = heads, rows >= G are zero. For an fp32 query, `lo` carries the remainder
// q - bf16(q) as a second set of bf16 fragments (zero for a bf16 query).
template <int D, int G>
__device__ __forceinline__ void load_q_frags(const void *q, size_t orow0, bool q32, uint32_t (&hi)[D / 16][2],
                                             uint32_t (&lo)[D / 16][2]) {
  const int lane = threadIdx.x & 31;
  const int hrow = lane >> 2, qcol = 2 * (lane & 3);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      hi[kk][j] = 0u;
      lo[kk][j] = 0u;
      if (hrow < G) {
        const size_t idx = (orow0 + hrow) * D + kk * 16 + j * 8 + qcol;
        if (!q32) {
          hi[kk][j] = *reinterpret_cast<const uint32_t *>(static_cast<const uint16_t *>(q) + idx);
        } else {
          const float2 qf = *reinterpret_cast<const float2 *>(static_cast<const float *>(q) + idx);
          hi[kk][j] = pack_bf16(qf.x, qf.y);
          lo[kk][j] = pack_bf16(qf.x - bf16_lo_f(hi[kk][j]), qf.y - bf16_hi_f(hi[kk][j]));
        }
      }
    }
}

// One 16-token page of K and V (swizzled tiles in shared memory, kpg and vpg) into a
// warp's online softmax state, with the tokens as the MMA rows and the heads as its
// columns (m16n8k16, bf16 inputs, fp32 accumulation; up to 8 heads):
//   S^T = K q^T      A = the page's K tile (16 tokens x 16 dims per k-step, ldmatrix),
//                    B = q^T (qa_hi / qa_lo: the query fragments of load_q_frags);
//   O^T += V^T P^T   A = V^T (16 dims x 16 tokens, transposed ldmatrix),
//                    B = P^T (the probabilities transposed in registers with movmatrix).
// P enters as a bf16 pair hi + lo (hi = bf16(p), lo = bf16(p - hi)), which keeps it to
// about 2^-16 relative. Each thread holds the state of heads h = 2(lane%4) + {0, 1}:
// m_run[], l_run[] (log2 units; replicated over the 8 lanes with equal lane%4) and
// o[m][j] = O[head h(j)][dim 16m + lane/4 + 8 (j >> 1)], j = (j & 1) picking the head.
// `valid` tokens (1..16) hold data: rows past it are zeroed in V and masked out of S.
// Scores in log2 units (qk_scale = log2(e) / sqrt(d)); bias2 (log2 units) is added to
// the score of every token of the page (0 for plain attention, -inf drops the page).
// Called by all 32 lanes.
template <int D>
__device__ __forceinline__ void mma_page(unsigned char *kpg, unsigned char *vpg, int valid,
                                         const uint32_t (&qa_hi)[D / 16][2], const uint32_t (&qa_lo)[D / 16][2],
                                         bool q32, float qk_scale, float bias2, float (&m_run)[2],
                                         float (&l_run)[2], float (&o)[D / 16][4]) {
  constexpr int KSTEPS = D / 16;
  const int lane = threadIdx.x & 31;
  if (valid < kPage) {
    // Rows past T may hold anything (even NaN): zero them in V; their scores are
    // masked below.
    for (int i = lane; i < (kPage - valid) * (D / 8); i += 32) {
      const int r = valid + i / (D / 8), c = i % (D / 8);
      *reinterpret_cast<uint4 *>(vpg + swz(r, c)) = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncwarp();
  }
  // ---- S^T = K q^T: two accumulators (even and odd k-steps) halve the MMA chain ---------
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
  const uint32_t kbase = smem_u32(kpg);
  const int lrow = ((lane >> 4) << 3) + (lane & 7);   // token row this lane addresses
  const int lsub = (lane >> 3) & 1;                  // low / high 8 columns of the k-step
#pragma unroll
  for (int kk = 0; kk < KSTEPS; ++kk) {
    uint32_t b0, b1, b2, b3;   // (tokens 0-7, cols 0-7), (0-7, 8-15), (8-15, 0-7), (8-15, 8-15)
    ldsm_x4(kbase + swz(lrow, 2 * kk + lsub), b0, b1, b2, b3);
    float (&acc)[4] = (kk & 1) ? s1 : s0;
    mma_bf16(acc, b0, b2, b1, b3, qa_hi[kk][0], qa_hi[kk][1]);
    if (q32) mma_bf16(acc, b0, b2, b1, b3, qa_lo[kk][0], qa_lo[kk][1]);
  }
  // ---- online softmax per head over the 16 tokens -----------------------------------
  // x[j]: token lane/4 + 8 (j >> 1), head 2(lane%4) + (j & 1).
  const int t0 = lane >> 2;
  float x[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int t = t0 + 8 * (j >> 1);
    x[j] = t < valid ? (s0[j] + s1[j]) * qk_scale + bias2 : -INFINITY;
  }
  float mx[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
#pragma unroll
  for (int o2 = 4; o2 < 32; o2 <<= 1) {
    mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], o2));
    mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xffffffffu, mx[1], o2));
  }
  float alpha[2], p[4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float m_new = fmaxf(m_run[h], mx[h]);
    alpha[h] = m_new == -INFINITY ? 1.0f : exp2f(m_run[h] - m_new);
    p[h] = m_new == -INFINITY ? 0.0f : exp2f(x[h] - m_new);
    p[h + 2] = m_new == -INFINITY ? 0.0f : exp2f(x[h + 2] - m_new);
    m_run[h] = m_new;
  }
  float ps[2] = {p[0] + p[2], p[1] + p[3]};
#pragma unroll
  for (int o2 = 4; o2 < 32; o2 <<= 1) {
    ps[0] += __shfl_xor_sync(0xffffffffu, ps[0], o2);
    ps[1] += __shfl_xor_sync(0xffffffffu, ps[1], o2);
  }
  l_run[0] = l_run[0] * alpha[0] + ps[0];
  l_run[1] = l_run[1] * alpha[1] + ps[1];
#pragma unroll
  for (int m = 0; m < D / 16; ++m) {
    o[m][0] *= alpha[0];
    o[m][1] *= alpha[1];
    o[m][2] *= alpha[0];
    o[m][3] *= alpha[1];
  }
  // P^T as bf16 hi + lo B fragments: pack (token, head pair) rows, transpose the two 8x8
  // blocks (tokens 0-7 and 8-15).
  const uint32_t ph0 = pack_bf16(p[0], p[1]), ph1 = pack_bf16(p[2], p[3]);
  const uint32_t pl0 = pack_bf16(p[0] - bf16_lo_f(ph0), p[1] - bf16_hi_f(ph0));
  const uint32_t pl1 = pack_bf16(p[2] - bf16_lo_f(ph1), p[3] - bf16_hi_f(ph1));
  const uint32_t bh0 = movmatrix_t(ph0), bh1 = movmatrix_t(ph1);
  const uint32_t bl0 = movmatrix_t(pl0), bl1 = movmatrix_t(pl1);
  // ---- O^T += V^T P^T: V^T fragments by transposed ldmatrix ------------------------------
  const uint32_t vbase = smem_u32(vpg);
  const int vrow = (lane & 7) + ((lane >> 4) << 3);  // token row this lane addresses
  const int vsub = (lane >> 3) & 1;                  // which 8-dim half of the m-tile
#pragma unroll
  for (int m = 0; m < D / 16; ++m) {
    uint32_t a0, a1, a2, a3;   // V^T (dims 0-7, tokens 0-7), (8-15, 0-7), (0-7, 8-15), (8-15, 8-15)
    ldsm_x4_t(vbase + swz(vrow, 2 * m + vsub), a0, a1, a2, a3);
    mma_bf16(o[m], a0, a1, a2, a3, bh0, bh1);
    mma_bf16(o[m], a0, a1, a2, a3, bl0, bl1);
  }
}

// A warp's softmax state (after mma_page) into shared memory: m and l of heads < G at
// mw[h], lw[h] (lanes 0-3 write).
template <int G>
__device__ __forceinline__ void store_warp_ml(const float (&m_run)[2], const float (&l_run)[2], float *mw, float *lw) {
  const int lane = threadIdx.x & 31;
  if (lane < 4) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int h = 2 * lane + j;
      if (h < G) {
        mw[h] = m_run[j];
        lw[h] = l_run[j];
      }
    }
  }
}
// A warp's O of heads < G into ow[h * D + d]: o * wt[h], added (fmaf) to what is there
// when `accumulate`; wt = null stores o as it is.
template <int D, int G>
__device__ __forceinline__ void add_warp_o(const float (&o)[D / 16][4], const float *wt, float *ow, bool accumulate) {
  const int lane = threadIdx.x & 31;
  const int h0 = 2 * (lane & 3), d0 = lane >> 2;
#pragma unroll
  for (int m = 0; m < D / 16; ++m)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int h = h0 + (j & 1), d = 16 * m + d0 + 8 * (j >> 1);
      if (h < G) {
        float *dst = ow + h * D + d;
        *dst = wt == nullptr ? o[m][j] : fmaf(o[m][j], wt[h], accumulate ? *dst : 0.0f);
      }
    }
}

// Returns false for a split that took no part (it left at once; see step_ws_splits).
template <int D, int G>
__device__ bool attn_split_mma(const AttnArgs &a, const CUtensorMap *tmk, const CUtensorMap *tmv, unsigned char *smem,
                               bool in_step, bool in_cluster) {
  using L = MmaLayout<D>;
  constexpr int NT = kMmaThreads;
  constexpr int KSTEPS = D / 16;
  const int R = attn_mma_ring(in_cluster);
  __shared__ uint64_t bars[L::kRingMax];
  __shared__ int slot_valid[L::kRingMax][kStagePages];
  __shared__ float slot_bias[L::kRingMax][kStagePages];   // log2 units, 0 without biases
  const bs_dims &dims = a.dims;
  int32_t *st = a.st;

  const int u = attn_unit_id(in_cluster), split = attn_split_id(in_cluster);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = u / dims.n_kv_heads, hk = u % dims.n_kv_heads;
  const size_t orow0 = static_cast<size_t>(b) * dims.n_q_heads + static_cast<size_t>(hk) * G;
  int32_t *sel_sm = reinterpret_cast<int32_t *>(smem + L::off_sel(R));
  const int n_part = in_step && !in_cluster ? step_ws_splits(a, u, attn_n_splits(false)) : attn_n_splits(in_cluster);
  if (split >= n_part) return false;

  prefetch_page_row<NT>(dims, a.kv, a.cfg, a.plist, u, in_step);
  UnitBlocks ub = load_unit_blocks<NT>(a, u, sel_sm, in_step, in_cluster);
  check_split_bound(ub, n_part, split, st);
  // Every split taking part stays to the end (an idle one with an empty state): the
  // merge needs all CTAs of a cluster (all launched ones take part there), and in
  // workspace mode the last split to arrive merges, after every split taking part has
  // read the unit's words.
  const int n_pages = ub.ok ? ub.pg.n_pages : 0;
  const int gp0 = min(split * ub.pg.pps, n_pages);
  const int gp1 = min(gp0 + ub.pg.pps, n_pages);
  const int n_stages = (gp1 - gp0 + kStagePages - 1) / kStagePages;
  const int32_t *pt = a.kv.page_table + static_cast<size_t>(u) * dims.max_pages_per_unit;

  if (tid == 0) {
    for (int i = 0; i < R; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Warp 0 resolves the split's pages 32 at a time (lane l: page 32 c + l of the split;
  // one round of page-table loads per chunk) and starts the copies of a stage's 4
  // pages (one TMA box per 64-column half of a page, for K and for V).
  int chunk = -1, ch_phys = -1, ch_valid = 0;
  float ch_bias = 0.0f;
  auto issue = [&](int stage, int buf) {
    const int first = stage * kStagePages;  // stages never straddle a chunk
    if (first / 32 != chunk) {
      chunk = first / 32;
      int blk = -1;
      ch_valid = resolve_page(ub, dims, pt, gp0 + chunk * 32 + lane, gp1, &ch_phys, a.bias ? &blk : nullptr, st);
      ch_bias = block_bias2(a.bias, dims, u, blk, st);
    }
    const int src = first - chunk * 32 + (lane & (kStagePages - 1));
    const int phys_l = __shfl_sync(0xffffffffu, ch_phys, src);
    const int valid_l = __shfl_sync(0xffffffffu, ch_valid, src);
    const float bias_l = __shfl_sync(0xffffffffu, ch_bias, src);
    const int phys = lane < kStagePages ? phys_l : -1;
    const int valid_tok = lane < kStagePages ? valid_l : 0;
    const unsigned m = __ballot_sync(0xffffffffu, valid_tok > 0);
    if (lane == 0) mbar_arrive_expect_tx(&bars[buf], static_cast<uint32_t>(__popc(m)) * 2u * L::kPageBytes);
    __syncwarp();
    if (valid_tok > 0) {
      fence_proxy_async_smem();
      unsigned char *kdst = smem + buf * L::kBufBytes + lane * L::kPageBytes;
      unsigned char *vdst = kdst + L::kStageKV;
#pragma unroll
      for (int hh = 0; hh < L::kHalves; ++hh) {
        tma_load_2d(kdst + hh * L::kHalfBytes, tmk, hh * 64, phys * kPage, &bars[buf]);
        tma_load_2d(vdst + hh * L::kHalfBytes, tmv, hh * 64, phys * kPage, &bars[buf]);
      }
    }
    if (lane < kStagePages) {
      slot_valid[buf][lane] = valid_tok;
      slot_bias[buf][lane] = bias_l;
    }
  };
  if (warp == 0)
    for (int i = 0; i < R && i < n_stages; ++i) issue(i, i);

  // Query rows as MMA A fragments (rows = heads; rows >= G are zero). For an fp32
  // query a second bf16 fragment carries the remainder q - bf16(q).
  const bool q32 = dims.q_dtype == BS_FP32;
  uint32_t qa_hi[KSTEPS][2], qa_lo[KSTEPS][2];
  load_q_frags<D, G>(a.q, orow0, q32, qa_hi, qa_lo);
  const float qk_scale = rsqrtf(static_cast<float>(D)) * kLog2e;

  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};   // heads 2(lane%4) + {0, 1}
  float o[D / 16][4];
#pragma unroll
  for (int m = 0; m < D / 16; ++m) o[m][0] = o[m][1] = o[m][2] = o[m][3] = 0.0f;

  int failed_at = -1;
  for (int it = 0; it < n_stages; ++it) {
    const int buf = it % R;
    const bool ok = mbar_wait_bounded(&bars[buf], static_cast<uint32_t>((it / R) & 1), st, a.wait_ns);
    // A copy that never lands: stop computing but still reach the merge (the status
    // word holds BS_ERR_TIMEOUT and the output is not meaningful).
    if (__syncthreads_or(!ok)) {
      failed_at = it;
      break;
    }
    const int valid = slot_valid[buf][warp];
    if (valid > 0) {
      unsigned char *kpg = smem + buf * L::kBufBytes + warp * L::kPageBytes;
      mma_page<D>(kpg, kpg + L::kStageKV, valid, qa_hi, qa_lo, q32, qk_scale, slot_bias[buf][warp], m_run, l_run,
                  o);
    }
    __syncthreads();
    if (warp == 0 && it + R < n_stages) issue(it + R, buf);
  }
  if (failed_at >= 0) {
    // Stages failed_at .. failed_at + R - 1 were issued and not consumed: wait (bounded)
    // for their copies before the buffers are reused below or the CTA exits.
    if (tid == 0)
      for (int s2 = failed_at; s2 < min(n_stages, failed_at + R); ++s2)
        mbar_wait_bounded(&bars[s2 % R], static_cast<uint32_t>((s2 / R) & 1), st, a.wait_ns);
    __syncthreads();
  }

  // ---- combine the four warps' states ---------------------------------------------
  float *ow = reinterpret_cast<float *>(smem);               // [4][8][D] in buffer 0
  float *mw = ow + 4 * kMaxG * D;                            // [4][8]
  float *lw = mw + 4 * kMaxG;                                // [4][8]
  add_warp_o<D, G>(o, nullptr, ow + warp * kMaxG * D, false);
  store_warp_ml<G>(m_run, l_run, mw + warp * kMaxG, lw + warp * kMaxG);
  __syncthreads();
  __shared__ float mfin[kMaxG], lfin[kMaxG], wfin[4][kMaxG];
  if (tid < G) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, mw[w * kMaxG + tid]);
    float Ls = 0.0f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float mi = mw[w * kMaxG + tid];
      const float wt = (mi == -INFINITY) ? 0.0f : exp2f(mi - M);
      wfin[w][tid] = wt;
      Ls = fmaf(lw[w * kMaxG + tid], wt, Ls);
    }
    mfin[tid] = M;
    lfin[tid] = Ls;
  }
  __syncthreads();
  float *osum = reinterpret_cast<float *>(smem + L::kBufBytes);   // [G][D] in buffer 1
  for (int i = tid; i < G * D / 4; i += NT) {
    const int h = i / (D / 4), dq = i % (D / 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float wt = wfin[w][h];
      const float4 v = reinterpret_cast<const float4 *>(ow + (w * kMaxG + h) * D)[dq];
      acc.x = fmaf(v.x, wt, acc.x);
      acc.y = fmaf(v.y, wt, acc.y);
      acc.z = fmaf(v.z, wt, acc.z);
      acc.w = fmaf(v.w, wt, acc.w);
    }
    reinterpret_cast<float4 *>(osum + h * D)[dq] = acc;
  }
  __syncthreads();
  if (in_cluster) {
    cluster_merge<NT, D, G>(orow0, osum, mfin, lfin, a.out, a.lse);
    // Every CTA of the cluster has read the unit's words: advance its epoch.
    if (ub.polled && split == 0 && tid == 0) a.expect[u] = ub.epoch;
  } else {
    finish_split<NT, D, G>(ub, u, orow0, osum, mfin, lfin, a.arrivals, a.records, a.out, a.lse,
                           reinterpret_cast<float *>(smem + L::kBufBytes + G * D * 4), a.expect, n_part);
  }
  return true;
}

// ===========================================================================
// fp32 path: 1-D bulk copies + FFMA
// ===========================================================================
constexpr int kFfmaThreads = 256;  // 8 warps

template <int D, int G>
struct FfmaLayout {
  static constexpr int kPageBytes = kPage * D * 4;
  static constexpr int kStageBytes = kStagePages * kPageBytes;
  static constexpr int kGP = (G + 3) & ~3;  // p row stride (floats)
  static constexpr int kOffQ = 4 * kStageBytes;
  static constexpr int kOffS = kOffQ + G * D * 4;
  static constexpr int kOffP = kOffS + G * kStageTokens * 4;
  static constexpr int kOffA = kOffP + kStageTokens * kGP * 4;
  static constexpr int kOffSel = kOffA + kMaxG * 4;
  static constexpr int kBytes = kOffSel + kSelPreload * 4;
  static_assert(2 * kStageBytes >= 8 * G * D * 4 + G * D * 4, "reduction scratch must fit in the K stages");
  static_assert(2 * kStageBytes >= 3 * kMaxG * kAttnMaxSplits * 4, "merge scratch must fit in the V stages");
};

// Returns false for a split that took no part (it left at once; see step_ws_splits).
template <int D, int G>
__device__ bool attn_split_ffma(const AttnArgs &a, unsigned char *smem, bool in_step, bool in_cluster) {
  using L = FfmaLayout<D, G>;
  const bs_dims &dims = a.dims;
  const bs_kv &kv = a.kv;
  const void *q = a.q;
  int32_t *st = a.st;
  constexpr int NT = kFfmaThreads;
  constexpr int DPL = D / 32;
  constexpr int kPer = D / 16;  // 16-byte chunks per quarter of a row (fp32: D/4 chunks per row)
  __shared__ uint64_t bars[2];
  __shared__ int slot_valid[2][kStagePages];
  __shared__ float slot_bias[2][kStagePages];   // log2 units, 0 without biases
  __shared__ float ml_sm[2][kMaxG];

  const int u = attn_unit_id(in_cluster), split = attn_split_id(in_cluster);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = u / dims.n_kv_heads, hk = u % dims.n_kv_heads;
  const size_t orow0 = static_cast<size_t>(b) * dims.n_q_heads + static_cast<size_t>(hk) * G;
  int32_t *sel_sm = reinterpret_cast<int32_t *>(smem + L::kOffSel);
  const int n_part = in_step && !in_cluster ? step_ws_splits(a, u, attn_n_splits(false)) : attn_n_splits(in_cluster);
  if (split >= n_part) return false;

  prefetch_page_row<NT>(dims, kv, a.cfg, a.plist, u, in_step);
  UnitBlocks ub = load_unit_blocks<NT>(a, u, sel_sm, in_step, in_cluster);
  check_split_bound(ub, n_part, split, st);
  // Every split taking part stays to the end (see attn_split_mma).
  const int n_pages = ub.ok ? ub.pg.n_pages : 0;
  const int gp0 = min(split * ub.pg.pps, n_pages);
  const int gp1 = min(gp0 + ub.pg.pps, n_pages);
  const int n_stages = (gp1 - gp0 + kStagePages - 1) / kStagePages;
  const int32_t *pt = kv.page_table + static_cast<size_t>(u) * dims.max_pages_per_unit;
  const unsigned char *kpool = static_cast<const unsigned char *>(kv.k_pool);
  const unsigned char *vpool = static_cast<const unsigned char *>(kv.v_pool);

  float *qs = reinterpret_cast<float *>(smem + L::kOffQ);
  float *s_sm = reinterpret_cast<float *>(smem + L::kOffS);
  float *p_sm = reinterpret_cast<float *>(smem + L::kOffP);
  float *alpha_sm = reinterpret_cast<float *>(smem + L::kOffA);

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncthreads();

  auto issue = [&](int stage, int buf) {
    int phys = -1, valid_tok = 0, blk = -1;
    if (lane < kStagePages)
      valid_tok = resolve_page(ub, dims, pt, gp0 + stage * kStagePages + lane, gp1, &phys, a.bias ? &blk : nullptr, st);
    const float bias2 = lane < kStagePages ? block_bias2(a.bias, dims, u, blk, st) : 0.0f;
    const unsigned m = __ballot_sync(0xffffffffu, valid_tok > 0);
    if (lane == 0) mbar_arrive_expect_tx(&bars[buf], static_cast<uint32_t>(__popc(m)) * 2u * L::kPageBytes);
    __syncwarp();
    if (valid_tok > 0) {
      fence_proxy_async_smem();
      const size_t src = static_cast<size_t>(phys) * L::kPageBytes;
      bulk_g2s(smem + buf * L::kStageBytes + lane * L::kPageBytes, kpool + src, L::kPageBytes, &bars[buf]);
      bulk_g2s(smem + (2 + buf) * L::kStageBytes + lane * L::kPageBytes, vpool + src, L::kPageBytes, &bars[buf]);
    }
    if (lane < kStagePages) {
      slot_valid[buf][lane] = valid_tok;
      slot_bias[buf][lane] = bias2;
    }
  };

  if (warp == 0) {
    if (n_stages > 0) issue(0, 0);
    if (n_stages > 1) issue(1, 1);
  }
  {
    const float qscale = rsqrtf(static_cast<float>(D)) * kLog2e;
    const size_t qbase = orow0 * D;
    for (int i = tid; i < G * D; i += NT) qs[i] = load_scalar(q, qbase + i, dims.q_dtype) * qscale;
  }

  float m_run = -INFINITY, l_run = 0.0f;
  float acc[G][DPL];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int j = 0; j < DPL; ++j) acc[h][j] = 0.0f;

  const int tok = tid >> 2, qq = tid & 3;
  int failed_at = -1;
  for (int it = 0; it < n_stages; ++it) {
    const int buf = it & 1;
    const bool ok = mbar_wait_bounded(&bars[buf], static_cast<uint32_t>((it >> 1) & 1), st, a.wait_ns);
    if (__syncthreads_or(!ok)) {
      failed_at = it;
      break;
    }

    const unsigned char *Kb = smem + buf * L::kStageBytes;
    const bool tvalid = (tok & (kPage - 1)) < slot_valid[buf][tok >> 4];
    float a[G];
#pragma unroll
    for (int h = 0; h < G; ++h) a[h] = 0.0f;
    if (tvalid) {
      const float4 *row = reinterpret_cast<const float4 *>(Kb + tok * D * 4);
#pragma unroll
      for (int c = 0; c < kPer; ++c) {
        const int ch = qq + 4 * ((c + tok) & (kPer - 1));
        const float4 k4 = row[ch];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 q4 = reinterpret_cast<const float4 *>(qs + h * D)[ch];
          a[h] = fmaf(q4.x, k4.x, a[h]);
          a[h] = fmaf(q4.y, k4.y, a[h]);
          a[h] = fmaf(q4.z, k4.z, a[h]);
          a[h] = fmaf(q4.w, k4.w, a[h]);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      a[h] += __shfl_xor_sync(0xffffffffu, a[h], 1);
      a[h] += __shfl_xor_sync(0xffffffffu, a[h], 2);
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
      if ((h & 3) == qq) s_sm[h * kStageTokens + tok] = tvalid ? a[h] + slot_bias[buf][tok >> 4] : -INFINITY;
    __syncthreads();

    if (warp < G) {
      const float s0 = s_sm[warp * kStageTokens + lane];
      const float s1 = s_sm[warp * kStageTokens + lane + 32];
      float mx = fmaxf(s0, s1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(m_run, mx);
      float alpha = 1.0f, p0 = 0.0f, p1 = 0.0f;
      if (m_new != -INFINITY) {
        alpha = exp2f(m_run - m_new);
        p0 = exp2f(s0 - m_new);
        p1 = exp2f(s1 - m_new);
      }
      float ps = p0 + p1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l_run = l_run * alpha + ps;
      m_run = m_new;
      p_sm[lane * L::kGP + warp] = p0;
      p_sm[(lane + 32) * L::kGP + warp] = p1;
      if (lane == 0) alpha_sm[warp] = alpha;
    }
    __syncthreads();

    {
      float al[G];
#pragma unroll
      for (int h = 0; h < G; ++h) al[h] = alpha_sm[h];
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int j = 0; j < DPL; ++j) acc[h][j] *= al[h];
      const float *Vb = reinterpret_cast<const float *>(smem + (2 + buf) * L::kStageBytes);
#pragma unroll 2
      for (int i = 0; i < kStageTokens / 8; ++i) {
        const int t = warp + 8 * i;
        if ((t & (kPage - 1)) >= slot_valid[buf][t >> 4]) continue;  // warp-uniform
        float v[DPL];
#pragma unroll
        for (int j = 0; j < DPL; ++j) v[j] = Vb[t * D + lane * DPL + j];
        float p[L::kGP];
#pragma unroll
        for (int h4 = 0; h4 < L::kGP / 4; ++h4) {
          const float4 pv = reinterpret_cast<const float4 *>(p_sm + t * L::kGP)[h4];
          p[4 * h4 + 0] = pv.x; p[4 * h4 + 1] = pv.y; p[4 * h4 + 2] = pv.z; p[4 * h4 + 3] = pv.w;
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int j = 0; j < DPL; ++j) acc[h][j] = fmaf(p[h], v[j], acc[h][j]);
      }
    }
    __syncthreads();
    if (warp == 0 && it + 2 < n_stages) issue(it + 2, buf);
  }
  if (failed_at >= 0) {
    // Wait (bounded) for the copies still in flight before the buffers are reused.
    if (tid == 0)
      for (int s2 = failed_at; s2 < min(n_stages, failed_at + 2); ++s2)
        mbar_wait_bounded(&bars[s2 & 1], static_cast<uint32_t>((s2 >> 1) & 1), st, a.wait_ns);
    __syncthreads();
  }

  // ---- sum the 8 warps' accumulators --------------------------------------------
  float *red = reinterpret_cast<float *>(smem);        // [8][G][D] over the K stages
  float *osum = red + 8 * G * D;                       // [G][D]
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int j = 0; j < DPL; ++j) red[(warp * G + h) * D + lane * DPL + j] = acc[h][j];
  if (warp < G && lane == 0) {
    ml_sm[0][warp] = m_run;
    ml_sm[1][warp] = l_run;
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += NT) {
    const int h = i / D, dd = i - h * D;
    float sum = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += red[(w * G + h) * D + dd];
    osum[h * D + dd] = sum;
  }
  __syncthreads();
  if (in_cluster) {
    cluster_merge<NT, D, G>(orow0, osum, ml_sm[0], ml_sm[1], a.out, a.lse);
    if (ub.polled && split == 0 && tid == 0) a.expect[u] = ub.epoch;
  } else {
    finish_split<NT, D, G>(ub, u, orow0, osum, ml_sm[0], ml_sm[1], a.arrivals, a.records, a.out, a.lse,
                           reinterpret_cast<float *>(smem + 2 * L::kStageBytes), a.expect, n_part);
  }
  return true;
}

}  // namespace bsi
