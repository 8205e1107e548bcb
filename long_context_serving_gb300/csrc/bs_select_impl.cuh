// Device code of the per-unit block selection (a3) and set-difference (a5), shared by
// the stand-alone kernels and the fused decode step.
//
// Selection: "Technische Samenvatting: Fluxion", Kerninzichten item 2 (streaming vs
// retrieval heads); "Technisches Resümee: NOSA", Methodik / 1. Algorithmus: NOSA,
// "Dual-Selection-Mechanismus" and "ED-DMA". Set-difference: NOSA, "2. System: NOSI".
//
// Keys are float32 values mapped to order-preserving uint32. The k-th largest key is
// found by a four-pass 8-bit radix select (histograms in shared memory, warp-aggregated
// with __match_any_sync); every key above it is taken, and of the keys equal to it the
// lowest block indices are taken (a prefix count in index order). The selection is
// written in ascending order by a compaction over block indices, so nothing is sorted.
#pragma once

#include "bs_internal.cuh"

namespace bsi {

// flag bits per block
constexpr uint8_t kSel = 1;     // in the final selection
constexpr uint8_t kAlive = 2;   // eligible for Gamma_e (dual)
constexpr uint8_t kEvict = 4;   // chosen by Gamma_e
constexpr uint8_t kElig = 8;    // eligible in the current top-k pass

template <int NT>
struct SelShared {
  static constexpr int kWarps = NT / 32;
  uint32_t hist[256];
  int warp_tot[kWarps];
  int bcast[4];
};

// Exclusive prefix sum of one int per thread over the CTA; *total gets the sum.
template <int NT>
__device__ __forceinline__ int block_excl_scan(int v, SelShared<NT> &sh, int *total) {
  constexpr int W = NT / 32;
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
    int w = lane < W ? sh.warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < W) sh.warp_tot[lane] = w;  // inclusive
  }
  __syncthreads();
  const int before = (warp > 0 ? sh.warp_tot[warp - 1] : 0) + x - v;
  *total = sh.warp_tot[W - 1];
  __syncthreads();
  return before;
}

// Marks with `mark` the k blocks of [lo, hi) carrying kElig with the largest keys
// (keys[c - lo]), lower index first among equal keys.
template <int NT>
__device__ void topk_mark(const uint32_t *keys, uint8_t *flags, int lo, int hi, int k, uint8_t mark,
                          SelShared<NT> &sh) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int n = hi - lo;
  if (k <= 0 || n <= 0) return;
  // Contiguous per-thread ranges keep the index order for the tie pass.
  const int per = (n + NT - 1) / NT;
  const int a = lo + tid * per, e = min(hi, a + per);
  int my = 0;
  for (int c = a; c < e; ++c) my += (flags[c] & kElig) ? 1 : 0;
  int n_elig;
  block_excl_scan<NT>(my, sh, &n_elig);
  if (k >= n_elig) {
    for (int c = a; c < e; ++c)
      if (flags[c] & kElig) flags[c] |= mark;
    __syncthreads();
    return;
  }
  uint32_t prefix = 0, pmask = 0;
  int rem = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += NT) sh.hist[i] = 0;
    __syncthreads();
    for (int base = lo; base < hi; base += NT) {
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
  int rank = block_excl_scan<NT>(eq, sh, &tot);
  for (int c = a; c < e; ++c) {
    if (!(flags[c] & kElig) || keys[c - lo] != prefix) continue;
    if (rank < rem) flags[c] |= mark;
    ++rank;
  }
  __syncthreads();
}

// Per-unit inputs of the selection.
struct SelUnit {
  int cls, k, k_e;
  Geom ge;
  const float *scores;   // row of unit u (candidates [c_lo, c_hi) are read)
  const float *evict;    // row of unit u, dual only
  uint8_t *alive;        // row of unit u, dual only
};

// Selects the blocks of one unit into `flags[0, n_blk)` (bit kSel). Uses keys[n_blk]
// and flags[n_blk] in shared memory. Reads scores with L2-only loads so that values
// written by other CTAs of the same grid are seen. All NT threads must call it.
template <int NT>
__device__ void select_unit_flags(const SelUnit &su, uint32_t *keys, uint8_t *flags, SelShared<NT> &sh) {
  const int tid = threadIdx.x;
  const Geom &ge = su.ge;
  const int lo = ge.c_lo, hi = ge.c_hi;
  for (int c = tid; c < ge.n_blk; c += NT) {
    const bool forced = c < ge.n_sink || c >= ge.local_lo;
    uint8_t f = forced ? kSel : 0;
    if (su.cls == BS_DUAL && c >= lo && c < hi && su.alive[c]) f |= kAlive;
    flags[c] = f;
  }
  __syncthreads();
  if (su.cls == BS_RETRIEVAL) {
    for (int c = lo + tid; c < hi; c += NT) {
      keys[c - lo] = order_key(__ldcg(su.scores + c));
      flags[c] |= kElig;
    }
    __syncthreads();
    topk_mark<NT>(keys, flags, lo, hi, su.k, kSel, sh);
  } else if (su.cls == BS_DUAL) {
    // Gamma_e: the k_e largest eviction logits among alive candidates.
    for (int c = lo + tid; c < hi; c += NT) {
      keys[c - lo] = order_key(su.evict[c]);
      if (flags[c] & kAlive) flags[c] |= kElig;
    }
    __syncthreads();
    topk_mark<NT>(keys, flags, lo, hi, su.k_e, kEvict, sh);
    // Strict eviction: candidates outside Gamma_e are dead from now on. Gamma_q: the
    // k - k_e largest scores among the candidates outside Gamma_e.
    for (int c = lo + tid; c < hi; c += NT) {
      const uint8_t f = flags[c];
      su.alive[c] = (f & kEvict) ? 1 : 0;
      keys[c - lo] = order_key(__ldcg(su.scores + c));
      flags[c] = static_cast<uint8_t>(((f & kEvict) ? kSel : kElig) | (f & kEvict));
    }
    __syncthreads();
    topk_mark<NT>(keys, flags, lo, hi, su.k - su.k_e, kSel, sh);
  }
}

// Ascending compaction of the flagged blocks into out[0, cap) (-1 padded) and, if
// given, into the shared list `copy`. Returns the count, or -1 when it exceeds cap
// (then the row is all -1).
template <int NT>
__device__ int compact_selection(const uint8_t *flags, int n_blk, int32_t *out, int cap, int32_t *copy,
                                 SelShared<NT> &sh) {
  const int tid = threadIdx.x;
  const int per = (n_blk + NT - 1) / NT;
  const int a = tid * per, e = min(n_blk, a + per);
  int mine = 0;
  for (int c = a; c < e; ++c) mine += (flags[c] & kSel) ? 1 : 0;
  int total;
  int pos = block_excl_scan<NT>(mine, sh, &total);
  if (total > cap) {
    for (int i = tid; i < cap; i += NT) out[i] = -1;
    return -1;
  }
  for (int c = a; c < e; ++c)
    if (flags[c] & kSel) {
      out[pos] = c;
      if (copy) copy[pos] = c;
      ++pos;
    }
  for (int i = total + tid; i < cap; i += NT) out[i] = -1;
  return total;
}

// ---------------------------------------------------------------------------
// Set-difference of two ascending lists held in shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool sorted_contains(const int32_t *v, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (v[mid] < x) lo = mid + 1;
    else hi = mid;
  }
  return lo < n && v[lo] == x;
}

// Writes the elements of a[0..na) missing from b[0..nb) to dst (ascending), pads
// with -1 up to cap and returns the count. All NT threads must call it.
template <int NT>
__device__ int sorted_diff_into(const int32_t *a, int na, const int32_t *b, int nb, int32_t *dst, int cap,
                                SelShared<NT> &sh) {
  const int tid = threadIdx.x;
  const int per = (na + NT - 1) / NT;
  const int s = tid * per, e = min(na, s + per);
  int mine = 0;
  for (int i = s; i < e; ++i) mine += sorted_contains(b, nb, a[i]) ? 0 : 1;
  int total;
  int before = block_excl_scan<NT>(mine, sh, &total);
  for (int i = s; i < e; ++i)
    if (!sorted_contains(b, nb, a[i])) dst[before++] = a[i];
  for (int i = total + tid; i < cap; i += NT) dst[i] = -1;
  return total;
}

}  // namespace bsi
