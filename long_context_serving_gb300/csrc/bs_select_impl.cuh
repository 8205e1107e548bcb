// Device code of the per-unit block selection (a3) and set-difference (a5), shared by
// the stand-alone kernels and the fused decode step.
//
// Selection: "Technische Samenvatting: Fluxion", Kerninzichten item 2 (streaming vs
// retrieval heads); "Technisches Resümee: NOSA", Methodik / 1. Algorithmus: NOSA,
// "Dual-Selection-Mechanismus" and "ED-DMA". Set-difference: NOSA, "2. System: NOSI".
//
// Keys are float32 values mapped to order-preserving uint32. topk_mark finds the top k
// with one min/max pass, one 2048-bucket histogram on (key - min) and an exact ranking
// of the boundary bucket; topk_mark_radix (a four-pass 8-bit radix select with
// warp-aggregated shared histograms) handles heavy ties. Ties go to the lowest block
// index. The selection is written in ascending order by a compaction over block
// indices, so nothing is sorted.
#pragma once

#include "bs_internal.cuh"

namespace bsi {

// flag bits per block
constexpr uint8_t kSel = 1;     // in the final selection
constexpr uint8_t kAlive = 2;   // eligible for Gamma_e (dual)
constexpr uint8_t kEvict = 4;   // chosen by Gamma_e
constexpr uint8_t kElig = 8;    // eligible in the current top-k pass

constexpr uint8_t kBnd = 16;    // in the boundary bucket of the fast top-k
constexpr int kBuckets = 2048;  // histogram buckets of the fast top-k
constexpr int kBndDirect = 256; // boundary buckets up to this size are ranked directly

template <int NT>
struct SelShared {
  static constexpr int kWarps = NT / 32;
  uint32_t hist[kBuckets];      // the radix passes use the first 256
  int warp_tot[kWarps];
  uint32_t warp_min[kWarps], warp_max[kWarps];
  int warp_cnt[kWarps];
  int bcast[4];
  int bnd_n;
  int bnd_idx[kBndDirect];
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

// Marks with `mark` the k blocks of [lo, hi) carrying `elig` with the largest keys
// (keys[c - lo]), lower index first among equal keys. Four-pass 8-bit radix select.
template <int NT>
__device__ __noinline__ void topk_mark_radix(const uint32_t *keys, uint8_t *flags, int lo, int hi, int k,
                                             uint8_t mark, SelShared<NT> &sh, uint8_t elig = kElig) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int n = hi - lo;
  if (k <= 0 || n <= 0) return;
  // Contiguous per-thread ranges keep the index order for the tie pass.
  const int per = (n + NT - 1) / NT;
  const int a = lo + tid * per, e = min(hi, a + per);
  int my = 0;
  for (int c = a; c < e; ++c) my += (flags[c] & elig) ? 1 : 0;
  int n_elig;
  block_excl_scan<NT>(my, sh, &n_elig);
  if (k >= n_elig) {
    for (int c = a; c < e; ++c)
      if (flags[c] & elig) flags[c] |= mark;
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
      if (c < hi && (flags[c] & elig)) {
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
    if (!(flags[c] & elig)) continue;
    const uint32_t key = keys[c - lo];
    if (key > prefix) flags[c] |= mark;
    else if (key == prefix) ++eq;
  }
  int tot;
  int rank = block_excl_scan<NT>(eq, sh, &tot);
  for (int c = a; c < e; ++c) {
    if (!(flags[c] & elig) || keys[c - lo] != prefix) continue;
    if (rank < rem) flags[c] |= mark;
    ++rank;
  }
  __syncthreads();
}

// Marks with `mark` the k blocks of [lo, hi) carrying kElig with the largest keys
// (keys[c - lo]), lower index first among equal keys; the same result as
// topk_mark_radix with fewer CTA barriers:
//   1. min, max and count of the eligible keys (one barrier);
//   2. a histogram over 2048 buckets of the float value placed linearly between the
//      minimum and the maximum, (x - min) * (2048 / (max - min)) in fp32 with round to
//      nearest: subtraction, multiplication by a positive constant and truncation are
//      each monotone, so every key in a bucket above the boundary bucket B is taken
//      and every key below is not;
//   3. a suffix count over the buckets finds B and how many of its keys are taken;
//   4. keys in B are ranked exactly by (key desc, index asc): directly when B holds
//      at most 256 keys, otherwise by the radix select restricted to B.
template <int NT>
__device__ __noinline__ void topk_mark(const uint32_t *keys, uint8_t *flags, int lo, int hi, int k, uint8_t mark,
                                       SelShared<NT> &sh) {
  constexpr int W = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = hi - lo;
  if (k <= 0 || n <= 0) return;
  const int per = (n + NT - 1) / NT;
  const int a = lo + tid * per, e = min(hi, a + per);
  // 1. min / max / count
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  int cnt = 0;
  for (int c = a; c < e; ++c)
    if (flags[c] & kElig) {
      const uint32_t key = keys[c - lo];
      kmin = min(kmin, key);
      kmax = max(kmax, key);
      ++cnt;
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  }
  if (lane == 0) {
    sh.warp_min[warp] = kmin;
    sh.warp_max[warp] = kmax;
    sh.warp_cnt[warp] = cnt;
  }
  for (int i = tid; i < kBuckets; i += NT) sh.hist[i] = 0;
  if (tid == 0) sh.bnd_n = 0;
  __syncthreads();
  kmin = 0xffffffffu;
  kmax = 0u;
  int n_elig = 0;
#pragma unroll
  for (int w = 0; w < W; ++w) {
    kmin = min(kmin, sh.warp_min[w]);
    kmax = max(kmax, sh.warp_max[w]);
    n_elig += sh.warp_cnt[w];
  }
  if (k >= n_elig || kmin == kmax) {
    // Everything is taken, or every key ties: the radix select settles it cheaply.
    topk_mark_radix<NT>(keys, flags, lo, hi, k, mark, sh);
    return;
  }
  // 2. histogram of the monotone bucket map
  // A zero, infinite or NaN range (equal keys, infinities) puts every key in bucket 0,
  // which the exact rank below still orders correctly.
  const float xmin = key_value(kmin);
  const float range = key_value(kmax) - xmin;
  float bscale = (range > 0.0f && range <= 3.0e38f) ? static_cast<float>(kBuckets) / range : 0.0f;
  if (!(bscale <= 3.0e38f)) bscale = 0.0f;  // a subnormal range
  auto bucket = [&](uint32_t key) -> uint32_t {
    if (bscale == 0.0f) return 0u;
    const float f = (key_value(key) - xmin) * bscale;  // in [0, 2048 (1 + eps)]
    return f >= static_cast<float>(kBuckets - 1) ? static_cast<uint32_t>(kBuckets - 1) : static_cast<uint32_t>(f);
  };
  for (int c = a; c < e; ++c)
    if (flags[c] & kElig) atomicAdd(&sh.hist[bucket(keys[c - lo])], 1u);
  __syncthreads();
  // 3. thread t owns buckets [kBuckets - bpt (t + 1), kBuckets - bpt t): suffix counts
  constexpr int bpt = kBuckets / NT;
  const int top = kBuckets - bpt * tid - 1;
  int mine = 0;
#pragma unroll
  for (int i = 0; i < bpt; ++i) mine += static_cast<int>(sh.hist[top - i]);
  int total;
  const int above = block_excl_scan<NT>(mine, sh, &total);
  if (above < k && k <= above + mine) {
    int run = above;
    for (int i = 0; i < bpt; ++i) {
      const int hcount = static_cast<int>(sh.hist[top - i]);
      if (run + hcount >= k) {
        sh.bcast[0] = top - i;    // boundary bucket B
        sh.bcast[1] = k - run;    // keys of B to take
        sh.bcast[2] = hcount;     // keys in B
        break;
      }
      run += hcount;
    }
  }
  __syncthreads();
  const uint32_t B = static_cast<uint32_t>(sh.bcast[0]);
  const int rem = sh.bcast[1], in_b = sh.bcast[2];
  // 4. take the buckets above B; collect B
  for (int c = a; c < e; ++c) {
    if (!(flags[c] & kElig)) continue;
    const uint32_t bk = bucket(keys[c - lo]);
    if (bk > B) flags[c] |= mark;
    else if (bk == B) {
      if (in_b <= kBndDirect) sh.bnd_idx[atomicAdd(&sh.bnd_n, 1)] = c;
      else flags[c] |= kBnd;
    }
  }
  __syncthreads();
  if (in_b <= kBndDirect) {
    for (int i = tid; i < in_b; i += NT) {
      const int c = sh.bnd_idx[i];
      const uint32_t key = keys[c - lo];
      int rank = 0;
      for (int j = 0; j < in_b; ++j) {
        const int c2 = sh.bnd_idx[j];
        const uint32_t k2 = keys[c2 - lo];
        rank += (k2 > key || (k2 == key && c2 < c)) ? 1 : 0;
      }
      if (rank < rem) flags[c] |= mark;
    }
    __syncthreads();
  } else {
    topk_mark_radix<NT>(keys, flags, lo, hi, rem, mark, sh, kBnd);
    for (int c = a; c < e; ++c) flags[c] &= static_cast<uint8_t>(~kBnd);
    __syncthreads();
  }
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
__device__ __noinline__ void select_unit_flags(const SelUnit &su, uint32_t *keys, uint8_t *flags, SelShared<NT> &sh) {
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
__device__ __noinline__ int compact_selection(const uint8_t *flags, int n_blk, int32_t *out, int cap, int32_t *copy,
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
// Set-difference of the new selection against the previous one, right after a
// selection: membership of a previous block in the new selection is its kSel flag;
// membership of a new block in the previous selection is a bit of `pbits` (one bit
// per block, n_words words of shared memory). One combined scan orders both outputs.
// cur[0, nc) and prev[0, np) are ascending lists in shared memory. All NT threads call
// it; writes added / removed (padded with -1 to cap) and returns (added, removed).
// ---------------------------------------------------------------------------
template <int NT>
__device__ __noinline__ int2 setdiff_after_select(const int32_t *cur, int nc, const int32_t *prev, int np,
                                                  const uint8_t *flags, int n_blk, uint32_t *pbits, int n_words,
                                                  int32_t *added, int32_t *removed, int cap, SelShared<NT> &sh) {
  const int tid = threadIdx.x;
  for (int i = tid; i < n_words; i += NT) pbits[i] = 0u;
  __syncthreads();
  for (int i = tid; i < np; i += NT) {
    const int c = prev[i];
    if (c >= 0 && c < n_words * 32) atomicOr(&pbits[c >> 5], 1u << (c & 31));
  }
  __syncthreads();
  const int pc = (nc + NT - 1) / NT, pp = (np + NT - 1) / NT;
  const int ca = tid * pc, ce = min(nc, ca + pc);
  const int pa = tid * pp, pe = min(np, pa + pp);
  int na = 0, nr = 0;
  for (int i = ca; i < ce; ++i) {
    const int c = cur[i];
    na += (pbits[c >> 5] >> (c & 31)) & 1u ? 0 : 1;
  }
  for (int i = pa; i < pe; ++i) {
    const int c = prev[i];
    nr += (c >= 0 && c < n_blk && (flags[c] & kSel)) ? 0 : 1;
  }
  int total;
  const int packed = block_excl_scan<NT>((na << 16) | nr, sh, &total);
  int wa = packed >> 16, wr = packed & 0xffff;
  for (int i = ca; i < ce; ++i) {
    const int c = cur[i];
    if (!((pbits[c >> 5] >> (c & 31)) & 1u)) added[wa++] = c;
  }
  for (int i = pa; i < pe; ++i) {
    const int c = prev[i];
    if (!(c >= 0 && c < n_blk && (flags[c] & kSel))) removed[wr++] = c;
  }
  const int ta = total >> 16, tr = total & 0xffff;
  for (int i = ta + tid; i < cap; i += NT) added[i] = -1;
  for (int i = tr + tid; i < cap; i += NT) removed[i] = -1;
  return make_int2(ta, tr);
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
