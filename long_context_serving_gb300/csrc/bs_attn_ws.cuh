// Sparse decode attention (a4), balanced mode: a persistent grid in which every CTA
// takes an equal share of the pages of all units ("Technische Samenvatting: Fluxion",
// Kerninzichten item 3: this work is bound by data movement, so the bytes are spread
// evenly over the GPU).
//
// The selected pages of every unit, in unit order, form one stream of W pages; CTA c
// takes pages [c W / P, (c + 1) W / P) of it (P CTAs, about two per SM), which may
// cover the end of one unit, whole units and the start of another: its "segments".
// Inside a CTA one producer warp and four consumer warps work through a ring of page
// slots with two mbarriers per slot:
//   * the producer resolves a segment's physical pages 32 at a time (page-table loads,
//     or the fused step's page list) and, as slots come free, starts for each page one
//     tiled TMA copy (128-byte swizzle) per 64-column half of K and of V, completing the
//     slot's "full" barrier with their byte count;
//   * consumer warp w takes pages w, w + 4, ... of each segment: waits for the slot's
//     full barrier, runs the page through its online softmax on tensor cores (mma_page),
//     and arrives on the slot's "empty" barrier so the producer can refill it. No
//     CTA-wide barrier per page: each warp runs at its own pace;
//   * at a segment's end the four consumer warps combine their states (a named barrier
//     among them only; the producer already streams the next segment's pages). A
//     segment that is a whole unit writes the output; otherwise it writes a split record
//     (o, m, l) to the workspace at index unit + CTA and takes the unit's arrival ticket,
//     and the last of the unit's segments merges its records in CTA order.
// The plan depends on every unit's page count: in a stand-alone call the counts of the
// selection; in the fused step the counts the selection will have, from each unit's
// geometry and budget (exact for streaming and retrieval units, an upper bound for dual
// ones), so the attention can be planned before the selection is published. A unit's
// pages in the fused step come from the page list its selection published; the
// producer waits (bounded) for that publication before resolving them, so the pages of
// units already selected stream while others are still being selected.
#pragma once

#include "bs_attn_impl.cuh"

namespace bsi {

constexpr int kWsConsumers = 3;
constexpr int kWsThreads = 32 * (kWsConsumers + 1);  // three consumer warps, then the producer

template <int D>
struct WsLayout {
  static constexpr int kPageBytes = MmaLayout<D>::kPageBytes;  // K (or V) of one page, swizzled halves
  static constexpr int kSlotBytes = 2 * kPageBytes;             // K, then V
  static constexpr int kSlots = D == 128 ? 12 : 24;             // ring of page slots (96 KB)
  static constexpr int kOffML = kSlots * kSlotBytes;            // consumer warps' m, l [2][3][8]
  static constexpr int kOffOsum = kOffML + 2 * kWsConsumers * kMaxG * 4;  // combined o [8][D]
  static constexpr int kOffPlan = kOffOsum + kMaxG * D * 4;     // unit page offsets [kWsMaxUnits + 1]
  static constexpr int kOffScratch = kOffPlan + (kWsMaxUnits + 1 + 3) / 4 * 16;  // merge w, l [2][8][64]
  static constexpr int kMergeBatch = 64;                        // records merged per pass
  static constexpr int kOffPages = kOffScratch + 2 * kMaxG * kMergeBatch * 4;  // resolved pages [kPageWin]
  static constexpr int kPageWin = 256;                          // pages resolved per round
  static constexpr int kOffBias = kOffPages + kPageWin * 4;     // their logit biases [kPageWin]
  static constexpr int kBytes = kOffBias + kPageWin * 4;        // two CTAs per SM
};

// A resolved page: physical page | ((valid tokens - 1) << 27), non-negative since pools
// hold fewer than 2^27 pages (the dims check) and a page holds 1..16 valid tokens; -1
// for no page.
__device__ __forceinline__ int ws_pack_page(int phys, int valid) {
  return valid > 0 ? phys | ((valid - 1) << 27) : -1;
}

constexpr int kWsMaxPending = 4;   // split records of a CTA whose ticket is checked at its end

// The CTA of a balanced launch that holds page p of the stream (W pages cut among
// P <= W CTAs, CTA c taking [floor(c W / P), floor((c + 1) W / P))): the largest c with
// floor(c W / P) <= p.
__device__ __forceinline__ int ws_cta_of(int p, int W, int P) {
  return static_cast<int>(((static_cast<int64_t>(p) + 1) * P + W - 1) / W) - 1;
}

// Pages planned for unit u. In the fused step (in_step) they come from the unit's
// geometry and budget before the selection exists: forced blocks plus min(k,
// candidates) for retrieval and dual units (Gamma_e may find fewer alive blocks, so this
// is an upper bound for dual units), the tail block (which holds token T-1) last. In a
// stand-alone call, from the selection count: count * g/16 pages, of which the partial
// tail block's pages past T stay empty. Either way the plan needs one round of loads
// and no selection entry. Reports and returns 0 for a unit whose configuration breaks a
// rule. `T`, `g` and the other inputs are the unit's, loaded by the caller.
__device__ __forceinline__ int ws_plan_pages(const AttnArgs &a, bool in_step, int T, int g, int cls, int s, int sink,
                                             int local, int k, int cnt) {
  const bs_dims &dims = a.dims;
  if (T < 1 || g <= 0 || g % kPage != 0) {
    report(a.st, BS_ERR_INVALID_ARG);
    return 0;
  }
  if (in_step) {
    if (s <= 0 || local < 1 || sink < 0) {
      report(a.st, BS_ERR_INVALID_ARG);
      return 0;
    }
    const Geom ge = unit_geom(T, g, s, sink, local);
    const int lo2 = ge.local_lo > ge.n_sink ? ge.local_lo : ge.n_sink;
    int n = ge.n_sink + (ge.n_blk - lo2);
    if (cls != BS_STREAMING) n += min(max(k, 0), ge.c_hi - ge.c_lo);
    if (n > dims.max_sel_per_unit) n = dims.max_sel_per_unit;
    return unit_pages(T, g, n, ge.n_blk - 1, 1, kStagePages).n_pages;
  }
  if (cnt < 0 || cnt > dims.max_sel_per_unit) {
    report(a.st, BS_ERR_INVALID_ARG);
    return 0;
  }
  return cnt * (g / kPage);
}

// Segment iteration over a CTA's page range [p0, p1) of the stream: unit u and its local
// pages [lp0, lp1), the stream index of the first.
struct WsSeg {
  int u, lp0, lp1, p_first;
};

// First unit whose pages end past p (binary search over the offsets; off[U] = W).
__device__ __forceinline__ int ws_first_unit(const int *off, int U, int p) {
  int lo = 0, hi = U - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (off[mid + 1] <= p) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// The segment that starts at stream page p (p0 <= p < p1), skipping empty units.
__device__ __forceinline__ WsSeg ws_segment_at(const int *off, int U, int p, int p1) {
  WsSeg sg;
  sg.u = ws_first_unit(off, U, p);
  sg.p_first = p;
  sg.lp0 = p - off[sg.u];
  sg.lp1 = min(p1, off[sg.u + 1]) - off[sg.u];
  return sg;
}

// Exclusive prefix sum over the CTA (NT threads, one value each), via shared `tmp`
// (NT/32 ints); *total gets the sum. All NT threads call it.
template <int NT>
__device__ __forceinline__ int ws_block_scan(int v, int *tmp, int *total) {
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
  for (int w = 0; w < NT / 32; ++w) {
    const int t = tmp[w];
    if (w < warp) before += t;
    tot += t;
  }
  __syncthreads();
  *total = tot;
  return before + x - v;
}

// Small shared state of a balanced CTA (the large buffers are in dynamic shared memory).
template <int NS>
struct WsShared {
  uint64_t full_bar[NS], empty_bar[NS];
  int slot_valid[NS];
  float slot_bias[NS];   // log2 units, 0 without biases
  int scan_tmp[kWsThreads / 32];
  int is_last, abort_flag;
  float mfin[kMaxG], lfin[kMaxG], wfin[kWsConsumers][kMaxG];
  int pend_u[kWsMaxPending];
};

// The CTA's share of the page stream: pages [p0, p1) of W, cut among Pe CTAs; off[u] the
// first page of unit u (off[U] = W).
struct WsPlan {
  const int *off;
  int U, W, Pe, p0, p1, c;
};

template <int D, int G>
__device__ __noinline__ void ws_producer(const AttnArgs &a, const CUtensorMap *tmk, const CUtensorMap *tmv,
                                         unsigned char *smem, WsShared<WsLayout<D>::kSlots> &sh, const WsPlan pl,
                                         bool in_step);
template <int D, int G>
__device__ __noinline__ void ws_consumer(const AttnArgs &a, unsigned char *smem, WsShared<WsLayout<D>::kSlots> &sh,
                                         const WsPlan pl, bool in_step);

template <int D, int G>
__device__ void attn_balanced_mma(const AttnArgs &a, const CUtensorMap *tmk, const CUtensorMap *tmv,
                                  unsigned char *smem, bool in_step) {
  using L = WsLayout<D>;
  constexpr int NS = L::kSlots;
  constexpr int QD = D / 4;
  __shared__ WsShared<NS> sh;
  uint64_t *full_bar = sh.full_bar, *empty_bar = sh.empty_bar;
  int *scan_tmp = sh.scan_tmp;
  const bs_dims &dims = a.dims;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int U = dims.batch * dims.n_kv_heads;
  const int P = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  int *off = reinterpret_cast<int *>(smem + L::kOffPlan);

  // ---- plan: every unit's pages, their offsets in the stream --------------------------
  {
    // Counts, four units per thread at a time with every load issued before any is used.
    constexpr int NB = 4;
    for (int u0 = tid; u0 < U; u0 += NB * kWsThreads) {
      int T[NB], g[NB], cls[NB], s[NB], sink[NB], local[NB], k[NB], cnt[NB];
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        const int u = u0 + j * kWsThreads;
        T[j] = g[j] = cls[j] = s[j] = sink[j] = local[j] = k[j] = cnt[j] = 0;
        if (u < U) {
          T[j] = a.kv.seq_lens[u / dims.n_kv_heads];
          g[j] = a.cfg.block_tokens[u];
          if (in_step) {
            cls[j] = a.cfg.cls[u];
            s[j] = a.cfg.sub_tokens[u];
            sink[j] = a.cfg.sink_tokens[u];
            local[j] = a.cfg.local_tokens[u];
            k[j] = a.cfg.k_total[u];
          } else {
            cnt[j] = __ldcg(a.sel_cnt + u);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        const int u = u0 + j * kWsThreads;
        if (u < U) off[u] = ws_plan_pages(a, in_step, T[j], g[j], cls[j], s[j], sink[j], local[j], k[j], cnt[j]);
      }
    }
    __syncthreads();
    // Exclusive prefix over the counts: contiguous chunks per thread, one block scan.
    const int per = (U + kWsThreads - 1) / kWsThreads;
    const int u0 = tid * per, u1 = min(U, u0 + per);
    int mine = 0;
    for (int u = u0; u < u1; ++u) mine += off[u];
    int total;
    int run = ws_block_scan<kWsThreads>(mine, scan_tmp, &total);
    for (int u = u0; u < u1; ++u) {
      const int n = off[u];
      off[u] = run;
      run += n;
    }
    if (tid == 0) {
      off[U] = total;
      sh.abort_flag = 0;
      for (int i = 0; i < NS; ++i) {
        mbar_init(&full_bar[i], 1);
        mbar_init(&empty_bar[i], 1);
      }
      fence_mbar_init();
    }
    __syncthreads();
  }
  // The stream is cut among P' = min(P, W) CTAs so that every share is non-empty: the
  // CTAs holding a unit's pages are then exactly c_first .. c_last.
  const int W = off[U];
  const int Pe = min(P, W);
  const int p0 = c < Pe ? static_cast<int>(static_cast<int64_t>(W) * c / Pe) : 0;
  const int p1 = c < Pe ? static_cast<int>(static_cast<int64_t>(W) * (c + 1) / Pe) : 0;
  // A unit with no pages at all (nothing to attend, or a broken rule) gets a zero row
  // and lse = -inf from one CTA.
  for (int u = tid; u < U; u += kWsThreads)
    if (off[u + 1] == off[u] && u % P == c) {
      const int b = u / dims.n_kv_heads, hk = u % dims.n_kv_heads;
      const size_t orow0 = static_cast<size_t>(b) * dims.n_q_heads + static_cast<size_t>(hk) * G;
      for (int i = 0; i < G * QD; ++i) {
        reinterpret_cast<float4 *>(a.out + (orow0 + i / QD) * D)[i % QD] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i % QD == 0) a.lse[orow0 + i / QD] = -INFINITY;
      }
    }
  if (p0 >= p1) return;
  const WsPlan pl{off, U, W, Pe, p0, p1, c};
  if (warp == kWsConsumers)
    ws_producer<D, G>(a, tmk, tmv, smem, sh, pl, in_step);
  else
    ws_consumer<D, G>(a, smem, sh, pl, in_step);
}

// The producer warp: resolves each segment's pages and starts their copies into the
// ring as slots come free.
template <int D, int G>
__device__ __noinline__ void ws_producer(const AttnArgs &a, const CUtensorMap *tmk, const CUtensorMap *tmv,
                                         unsigned char *smem, WsShared<WsLayout<D>::kSlots> &sh, const WsPlan pl,
                                         bool in_step) {
  using L = WsLayout<D>;
  constexpr int NS = L::kSlots;
  const bs_dims &dims = a.dims;
  int32_t *st = a.st;
  const int lane = threadIdx.x & 31;
  const int *off = pl.off;
  const int U = pl.U, p0 = pl.p0, p1 = pl.p1;
  uint64_t *full_bar = sh.full_bar, *empty_bar = sh.empty_bar;
  int *slot_valid = sh.slot_valid;
  float *slot_bias = sh.slot_bias;
  {
    int *pages = reinterpret_cast<int *>(smem + L::kOffPages);
    float *pbias = reinterpret_cast<float *>(smem + L::kOffBias);
    int last_use[NS];           // use index of each slot's latest page (-1: none)
#pragma unroll
    for (int i = 0; i < NS; ++i) last_use[i] = -1;
    for (int p = p0; p < p1;) {
      const WsSeg sg = ws_segment_at(off, U, p, p1);
      const int u = sg.u;
      const int b = u / dims.n_kv_heads;
      const int T = a.kv.seq_lens[b];
      const int g = a.cfg.block_tokens[u];
      const int ppb = g / kPage;
      const int32_t *pt = a.kv.page_table + static_cast<size_t>(u) * dims.max_pages_per_unit;
      const int cls = a.cfg.cls[u];
      // Pages of the unit that exist this step, and where they come from.
      int n_act = off[u + 1] - off[u];
      const int32_t *plist = nullptr;
      int n_sink = 0, lo2 = 0;
      const int32_t *sel = a.sel_idx + static_cast<size_t>(u) * dims.max_sel_per_unit;
      if (in_step && cls == BS_STREAMING) {
        const Geom ge = unit_geom(T, g, a.cfg.sub_tokens[u], a.cfg.sink_tokens[u], a.cfg.local_tokens[u]);
        n_sink = ge.n_sink;
        lo2 = ge.local_lo > ge.n_sink ? ge.local_lo : ge.n_sink;
      } else if (in_step) {
        int cnt = 0, e = 0;
        if (lane == 0) cnt = wait_published(a.pub, a.expect, u, a.wait_ns, st, &e);
        cnt = __shfl_sync(0xffffffffu, cnt, 0);
        n_act = cnt > 0 ? unit_pages(T, g, cnt, (T - 1) / g, 1, kStagePages).n_pages : 0;
        if (n_act > dims.max_gather_pages_per_unit) {
          if (lane == 0) report(st, BS_ERR_CAPACITY);
          n_act = 0;
        }
        plist = a.plist + static_cast<size_t>(u) * dims.max_gather_pages_per_unit;
      }
      for (int w0 = sg.lp0; w0 < sg.lp1; w0 += L::kPageWin) {
        const int w1 = min(sg.lp1, w0 + L::kPageWin);
        // Resolve pages [w0, w1) into shared memory: every lane issues all its loads of
        // one kind before using any of them (block index, then page-table entry).
        constexpr int R = L::kPageWin / 32;
        int blk[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int lp = w0 + lane + 32 * r;
          blk[r] = -1;
          if (lp < w1 && lp < n_act) {
            if (plist != nullptr) {
              blk[r] = __ldcg(plist + lp);      // already the physical page
            } else {
              const int i = lp / ppb;
              blk[r] = (in_step && cls == BS_STREAMING) ? (i < n_sink ? i : lo2 + (i - n_sink)) : __ldcg(sel + i);
            }
          }
        }
        if (a.bias != nullptr) {
          // The block of each page (from the selection when the pages came resolved)
          // and its logit bias.
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int lp = w0 + lane + 32 * r;
            if (lp >= w1) continue;
            int c = -1;
            if (lp < n_act) c = plist != nullptr ? __ldcg(sel + lp / ppb) : blk[r];
            pbias[lp - w0] = block_bias2(a.bias, dims, u, c, st);
          }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int lp = w0 + lane + 32 * r;
          if (lp >= w1) continue;
          int phys = -1, valid = 0;
          if (lp < n_act) {
            if (plist != nullptr) {
              phys = blk[r];
              valid = lp == n_act - 1 ? (T - 1) % kPage + 1 : kPage;
            } else {
              const int lpg = blk[r] * ppb + (lp - (lp / ppb) * ppb);
              const int t0 = lpg * kPage;
              if (blk[r] >= 0 && lpg < dims.max_pages_per_unit && t0 < T) {
                phys = __ldg(pt + lpg);
                valid = min(kPage, T - t0);
              } else if (!(blk[r] >= 0 && t0 >= T && lp / ppb == n_act / ppb - 1 && blk[r] * g < T)) {
                // (the last selected block may be the partial tail block: its pages past
                // T are planned but empty; anything else out of range is an error)
                report(st, BS_ERR_DEVICE_BOUNDS);
              }
            }
            if (valid > 0 && (phys < 0 || phys >= dims.n_pages)) {
              report(st, BS_ERR_DEVICE_BOUNDS);
              valid = 0;
            }
          }
          pages[lp - w0] = ws_pack_page(phys, valid);
        }
        __syncwarp();
        if (lane == 0) {
          for (int lp = w0; lp < w1; ++lp) {
            if (*reinterpret_cast<volatile int *>(&sh.abort_flag)) break;  // nothing more is issued
            const int pj = p + (lp - sg.lp0) - p0;
            const int slot = pj % NS;
            const int use = pj / NS;
            if (use > 0) mbar_wait_bounded(&empty_bar[slot], static_cast<uint32_t>((use - 1) & 1), st, a.wait_ns);
            const int e = pages[lp - w0];
            const int valid = e < 0 ? 0 : (e >> 27) + 1, phys = e & ((1 << 27) - 1);
            slot_valid[slot] = valid;
            slot_bias[slot] = a.bias != nullptr ? pbias[lp - w0] : 0.0f;
            last_use[slot] = use;
            mbar_arrive_expect_tx(&full_bar[slot], valid > 0 ? 2u * L::kPageBytes : 0u);
            if (valid > 0) {
              fence_proxy_async_smem();
              unsigned char *kdst = smem + slot * L::kSlotBytes;
#pragma unroll
              for (int hh = 0; hh < D / 64; ++hh) {
                tma_load_2d(kdst + hh * MmaLayout<D>::kHalfBytes, tmk, hh * 64, phys * kPage, &full_bar[slot]);
                tma_load_2d(kdst + L::kPageBytes + hh * MmaLayout<D>::kHalfBytes, tmv, hh * 64, phys * kPage,
                            &full_bar[slot]);
              }
            }
          }
        }
        __syncwarp();
      }
      p += sg.lp1 - sg.lp0;
    }
    // Copies that a consumer gave up on may still be in flight: wait for the phase of
    // each slot's latest page (immediately done when it was consumed; phases complete in
    // order, so every earlier copy into the slot has landed too) before the CTA can exit.
    if (lane == 0)
      for (int i = 0; i < NS; ++i)
        if (last_use[i] >= 0) mbar_wait_bounded(&full_bar[i], static_cast<uint32_t>(last_use[i] & 1), st, a.wait_ns);
  }
}

// The four consumer warps: each page through a warp's online softmax, then per segment
// the combine, the output or split record, and the merges this CTA has to do.
template <int D, int G>
__device__ __noinline__ void ws_consumer(const AttnArgs &a, unsigned char *smem, WsShared<WsLayout<D>::kSlots> &sh,
                                         const WsPlan pl, bool in_step) {
  using L = WsLayout<D>;
  constexpr int NS = L::kSlots;
  constexpr int NC = kWsConsumers;
  constexpr int KSTEPS = D / 16;
  constexpr int REC = attn_record_floats(D);
  constexpr int QD = D / 4;
  const bs_dims &dims = a.dims;
  int32_t *st = a.st;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int *off = pl.off;
  const int U = pl.U, W = pl.W, Pe = pl.Pe, p0 = pl.p0, p1 = pl.p1, c = pl.c;
  uint64_t *full_bar = sh.full_bar, *empty_bar = sh.empty_bar;
  int *slot_valid = sh.slot_valid;
  int &is_last = sh.is_last;
  int &abort_flag = sh.abort_flag;
  float *mfin = sh.mfin, *lfin = sh.lfin;
  float (*wfin)[kMaxG] = sh.wfin;
  int *pend_u = sh.pend_u;
  const bool q32 = dims.q_dtype == BS_FP32;
  const float qk_scale = rsqrtf(static_cast<float>(D)) * kLog2e;
  float *mw = reinterpret_cast<float *>(smem + L::kOffML);
  float *lw = mw + NC * kMaxG;
  float *osum = reinterpret_cast<float *>(smem + L::kOffOsum);
  float *scratch = reinterpret_cast<float *>(smem + L::kOffScratch);
  constexpr int NCT = NC * 32;   // consumer threads
  // Split records this CTA wrote: their unit and (thread 0) the ticket the atomic
  // returned; the tickets are looked at only at the end, so their latency is hidden.
  int pt0 = 0, pt1 = 0, pt2 = 0, pt3 = 0;   // (thread 0) each atomic writes its own register
  int n_pend = 0;
  auto merge_unit = [&](int u) {
    // The last piece of unit u merges the unit's records in CTA order:
    // M = max m_i, w_i = 2^(m_i - M), L = sum w_i l_i, o = sum w_i o_i / L.
    // The records' (m, l) come in one parallel round of loads per batch of kMergeBatch
    // records (one pass when the unit has at most that many pieces); then each thread
    // sums its (head, column) entries over the records, eight loads in flight at once.
    const int b = u / dims.n_kv_heads, hk = u % dims.n_kv_heads;
    const size_t orow0 = static_cast<size_t>(b) * dims.n_q_heads + static_cast<size_t>(hk) * G;
    const int c_first = ws_cta_of(off[u], W, Pe), c_last = ws_cta_of(off[u + 1] - 1, W, Pe);
    const int ns = c_last - c_first + 1;
    const float *base = a.records + static_cast<size_t>(u + c_first) * G * REC;
    float *w_sm = scratch;                          // [G][kMergeBatch]: m, then the weights
    float *l_sm = scratch + kMaxG * L::kMergeBatch; // [G][kMergeBatch]
    constexpr int NR = (kMaxG * QD + NCT - 1) / NCT;
    float4 acc[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    float M = -INFINITY, Lsum = 0.0f;   // thread tid < G: head tid
    if (ns > L::kMergeBatch) {
      // Many pieces: the maximum first, over batches.
      for (int s0 = 0; s0 < ns; s0 += L::kMergeBatch) {
        const int nb = min(L::kMergeBatch, ns - s0);
        for (int i = tid; i < G * nb; i += NCT) {
          const int h = i / nb, j = i % nb;
          w_sm[h * L::kMergeBatch + j] = __ldcg(base + (static_cast<size_t>(s0 + j) * G + h) * REC + D);
        }
        named_barrier(1, NCT);
        if (tid < G)
          for (int j = 0; j < nb; ++j) M = fmaxf(M, w_sm[tid * L::kMergeBatch + j]);
        named_barrier(1, NCT);
      }
    }
    for (int s0 = 0; s0 < ns; s0 += L::kMergeBatch) {
      const int nb = min(L::kMergeBatch, ns - s0);
      for (int i = tid; i < G * nb; i += NCT) {
        const int h = i / nb, j = i % nb;
        const float *r = base + (static_cast<size_t>(s0 + j) * G + h) * REC + D;
        w_sm[h * L::kMergeBatch + j] = __ldcg(r);
        l_sm[h * L::kMergeBatch + j] = __ldcg(r + 1);
      }
      named_barrier(1, NCT);
      if (tid < G) {
        if (ns <= L::kMergeBatch)
          for (int j = 0; j < nb; ++j) M = fmaxf(M, w_sm[tid * L::kMergeBatch + j]);
        mfin[tid] = M;
        for (int j = 0; j < nb; ++j) {
          const float mi = w_sm[tid * L::kMergeBatch + j];
          const float w = (mi == -INFINITY) ? 0.0f : exp2f(mi - M);
          w_sm[tid * L::kMergeBatch + j] = w;
          Lsum = fmaf(l_sm[tid * L::kMergeBatch + j], w, Lsum);
        }
      }
      named_barrier(1, NCT);
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const int i = tid + r * NCT;
        if (i < G * QD) {
          const int h = i / QD, dq = i % QD;
          const float4 *col = reinterpret_cast<const float4 *>(base + (static_cast<size_t>(s0) * G + h) * REC) + dq;
          const size_t stride = static_cast<size_t>(G) * REC / 4;    // float4s from one record to the next
          for (int j0 = 0; j0 < nb; j0 += 8) {
            float4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if (j0 + j < nb) v[j] = __ldcg(col + (j0 + j) * stride);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if (j0 + j < nb) {
                const float w = w_sm[h * L::kMergeBatch + j0 + j];
                acc[r].x = fmaf(v[j].x, w, acc[r].x);
                acc[r].y = fmaf(v[j].y, w, acc[r].y);
                acc[r].z = fmaf(v[j].z, w, acc[r].z);
                acc[r].w = fmaf(v[j].w, w, acc[r].w);
              }
          }
        }
      }
      named_barrier(1, NCT);
    }
    if (tid < G) lfin[tid] = Lsum;
    named_barrier(1, NCT);
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const int i = tid + r * NCT;
      if (i < G * QD) {
        const int h = i / QD, dq = i % QD;
        write_normalised(acc[r], mfin[h], lfin[h], a.out + (orow0 + h) * D, a.lse + orow0 + h, dq);
      }
    }
    if (tid == 0) {
      a.arrivals[u] = 0;  // ready for the next call
      if (in_step && a.cfg.cls[u] != BS_STREAMING) a.expect[u] = (__ldcg(a.expect + u) + 1) & kEpochMask;
    }
    named_barrier(1, NCT);
  };

  for (int p = p0; p < p1;) {
    const WsSeg sg = ws_segment_at(off, U, p, p1);
    const int u = sg.u;
    const int n = sg.lp1 - sg.lp0;
    const int b = u / dims.n_kv_heads, hk = u % dims.n_kv_heads;
    const size_t orow0 = static_cast<size_t>(b) * dims.n_q_heads + static_cast<size_t>(hk) * G;
    uint32_t qa_hi[KSTEPS][2], qa_lo[KSTEPS][2];
    load_q_frags<D, G>(a.q, orow0, q32, qa_hi, qa_lo);
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};   // heads 2(lane%4) + {0, 1}
    float o[D / 16][4];
#pragma unroll
    for (int m = 0; m < D / 16; ++m) o[m][0] = o[m][1] = o[m][2] = o[m][3] = 0.0f;
    for (int i = warp; i < n; i += NC) {
      const int pi = sg.p_first + i - p0;
      const int slot = pi % NS;
      const int use = pi / NS;
      // After a wait has given up (the copies of this CTA can no longer be trusted) the
      // remaining pages are skipped.
      const bool ok = !*reinterpret_cast<volatile int *>(&abort_flag) &&
                      mbar_wait_bounded(&full_bar[slot], static_cast<uint32_t>(use & 1), st, a.wait_ns);
      if (!ok && lane == 0) abort_flag = 1;
      const int valid = ok ? slot_valid[slot] : 0;
      if (valid > 0) {
        unsigned char *kpg = smem + slot * L::kSlotBytes;
        mma_page<D>(kpg, kpg + L::kPageBytes, valid, qa_hi, qa_lo, q32, qk_scale, sh.slot_bias[slot], m_run, l_run,
                    o);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[slot]);
    }
    // ---- combine the consumer warps' states of this segment --------------------------
    // M = max over warps, weights 2^(m_w - M); the warps add their weighted o into one
    // accumulator in warp order (fmaf, as a loop over the warps would).
    store_warp_ml<G>(m_run, l_run, mw + warp * kMaxG, lw + warp * kMaxG);
    named_barrier(1, NCT);
    if (tid < G) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NC; ++w) M = fmaxf(M, mw[w * kMaxG + tid]);
      float Ls = 0.0f;
#pragma unroll
      for (int w = 0; w < NC; ++w) {
        const float mi = mw[w * kMaxG + tid];
        const float wt = (mi == -INFINITY) ? 0.0f : exp2f(mi - M);
        wfin[w][tid] = wt;
        Ls = fmaf(lw[w * kMaxG + tid], wt, Ls);
      }
      mfin[tid] = M;
      lfin[tid] = Ls;
    }
    named_barrier(1, NCT);
#pragma unroll
    for (int w = 0; w < NC; ++w) {
      if (warp == w) add_warp_o<D, G>(o, wfin[w], osum, w > 0);
      named_barrier(1, NCT);
    }
    const bool whole = sg.lp0 == 0 && sg.lp1 == off[u + 1] - off[u];
    float *rec = a.records + static_cast<size_t>(u + c) * G * REC;
    for (int i = tid; i < G * QD; i += NCT) {
      const int h = i / QD, dq = i % QD;
      const float4 acc = reinterpret_cast<const float4 *>(osum + h * D)[dq];
      if (whole)   // the whole unit: write the output
        write_normalised(acc, mfin[h], lfin[h], a.out + (orow0 + h) * D, a.lse + orow0 + h, dq);
      else         // a piece: its split record (index unit + CTA)
        reinterpret_cast<float4 *>(rec + h * REC)[dq] = acc;
    }
    if (whole) {
      if (in_step && a.cfg.cls[u] != BS_STREAMING && tid == 0) a.expect[u] = (__ldcg(a.expect + u) + 1) & kEpochMask;
    } else {
      if (tid < G) {
        rec[tid * REC + D] = mfin[tid];
        rec[tid * REC + D + 1] = lfin[tid];
      }
      named_barrier(1, NCT);
      // The unit's arrival ticket (acquire-release: the record is published before it,
      // the last piece sees every record). Its value is looked at later.
      if (n_pend < kWsMaxPending) {
        if (tid == 0) {
          pend_u[n_pend] = u;
          switch (n_pend) {
            case 0: pt0 = atomic_add_acq_rel_gpu(a.arrivals + u, 1); break;
            case 1: pt1 = atomic_add_acq_rel_gpu(a.arrivals + u, 1); break;
            case 2: pt2 = atomic_add_acq_rel_gpu(a.arrivals + u, 1); break;
            default: pt3 = atomic_add_acq_rel_gpu(a.arrivals + u, 1); break;
          }
        }
        ++n_pend;
      } else {
        if (tid == 0) is_last = (atomic_add_acq_rel_gpu(a.arrivals + u, 1) ==
                                 ws_cta_of(off[u + 1] - 1, W, Pe) - ws_cta_of(off[u], W, Pe));
        named_barrier(1, NCT);
        if (is_last) merge_unit(u);
      }
    }
    named_barrier(1, NCT);   // the combine area is free for the next segment
    p += n;
  }
  // The units whose last piece this CTA wrote: merge them.
  for (int k = 0; k < n_pend; ++k) {
    if (tid == 0) {
      const int u = pend_u[k];
      const int t = k == 0 ? pt0 : k == 1 ? pt1 : k == 2 ? pt2 : pt3;
      is_last = t == ws_cta_of(off[u + 1] - 1, W, Pe) - ws_cta_of(off[u], W, Pe);
    }
    named_barrier(1, NCT);
    if (is_last) merge_unit(pend_u[k]);
    named_barrier(1, NCT);
  }
}

}  // namespace bsi
